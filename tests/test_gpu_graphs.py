"""The library's calls queue only stream work (kernels, memsets) and take
no host synchronisation, so a whole forward+backward can be captured into a
CUDA graph and replayed: the replay must give bit-identical results to the
eager calls, for both paths and both contraction variants, plain and with
a loss variant (label smoothing and z-loss)."""
import pytest
import torch

import chunked_lm_head_gemm_gb300 as lce
from chunked_lm_head_gemm_gb300.inputs import Workload, make_inputs
from tests.gpu_util import MODES, PAIRS, cta_pair, require_gpu

pytestmark = pytest.mark.gpu

WL = Workload("graph", 1000, 256, 5000, "bf16", 1.0, 0.05, "uniform",
              ignore_frac=0.1)


@pytest.mark.parametrize("variant", [{}, dict(label_smoothing=0.1,
                                                z_loss=1e-3)],
                         ids=["plain", "smoothing+zloss"])
@pytest.mark.parametrize("pair", PAIRS, ids=lambda v: "pair" if v else "cta")
@pytest.mark.parametrize("mode", MODES)
def test_captured_step_replays_bitwise(mode, pair, variant):
    dev = require_gpu()
    h, W, y = make_inputs(WL, seed=8, device=dev)
    L, H, V = WL.L, WL.H, WL.V
    chunk = 384
    ws = lce.alloc_workspace(L, H, V, h.dtype, chunk, dev)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    lse = torch.empty(L, dtype=torch.float32, device=dev)
    dH = torch.empty_like(h)
    dW = torch.empty(V, H, dtype=torch.float32, device=dev)
    dloss = torch.full((1,), 0.5, dtype=torch.float32, device=dev)

    def step():
        if mode == "fused":
            lce.forward_backward(h, W, y, chunk_rows=chunk, workspace=ws,
                                 loss_out=loss, lse_out=lse, dH_out=dH,
                                 dW_out=dW, **variant)
            lce.scale_gradients(dH, dW, dloss)
        else:
            lce.forward(h, W, y, workspace=ws, loss_out=loss, lse_out=lse,
                        **variant)
            lce.backward(h, W, y, lse, dloss, chunk_rows=chunk, workspace=ws,
                         dH_out=dH, dW_out=dW, **variant)

    with cta_pair(pair):
        step()                       # eager, also warms the library up
        torch.cuda.synchronize()
        ref = [t.clone() for t in (loss, lse, dH, dW)]
        for t in (loss, lse, dH, dW):
            t.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(2):
            for t in (loss, lse, dH, dW):
                t.zero_()
            g.replay()
            torch.cuda.synchronize()
            for got, want in zip((loss, lse, dH, dW), ref):
                assert torch.equal(got, want)
    assert lce.get_error() == 0
