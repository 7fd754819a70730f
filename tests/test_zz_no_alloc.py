"""lce_forward_static: the forward for callers that cannot allocate.

Some callers have no device allocator to give the library a workspace: a
runtime that owns all device memory and hands out only the tensors, code
that must not allocate after start-up, a plain C host. lce_forward_static
serves them from a fixed scratch array inside the library. This file checks,
through the C ABI, that it returns what lce_forward returns, on two calls in
a row of different sizes (the array keeps the previous call's contents, so
the second call must not depend on them), that it matches the float64
oracle, that it is right at its row limit (where the per-split partials
fill the array nearly to its end, and where a wide hidden size asks for
more column splits than the array holds, so the call uses fewer), and that
an L above its limit is refused before anything runs. It is collected last
on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from chunked_lm_head_gemm_gb300.inputs import Workload, make_inputs
from tests.gpu_util import LOSS_RTOL, LSE_ATOL, require_gpu

pytestmark = pytest.mark.gpu


def _static_forward(lib, h, W, y, ignore_index=-100):
    L, H = h.shape
    V = W.shape[0]
    loss = torch.empty((), dtype=torch.float32, device=h.device)
    lse = torch.empty(L, dtype=torch.float32, device=h.device)
    st = lib.lce_forward_static(
        ctypes.c_void_p(h.data_ptr()), ctypes.c_void_p(W.data_ptr()),
        ctypes.c_void_p(y.data_ptr()), L, H, V, ignore_index,
        ctypes.c_void_p(loss.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, loss, lse


def test_static_forward_matches_workspace_forward_twice():
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    lib = lce.load()
    cases = [Workload("static_a", 3000, 256, 20000, "bf16", 1.0, 0.05,
                      "uniform", ignore_frac=0.1),
             Workload("static_b", 700, 128, 5000, "bf16", 1.0, 0.1,
                      "uniform", ignore_frac=0.2)]
    for seed, wl in enumerate(cases):
        h, W, y = make_inputs(wl, seed=seed, device=dev)
        st, loss_s, lse_s = _static_forward(lib, h, W, y)
        assert st == 0, lib.lce_last_cuda_error().decode()
        loss_w, lse_w = lce.forward(h, W, y)
        assert lce.get_error() == 0
        ref = loss_w.item()
        assert abs(loss_s.item() - ref) <= LOSS_RTOL * abs(ref)
        err = np.max(np.abs(lse_s.cpu().double().numpy() -
                            lse_w.cpu().double().numpy()))
        assert err <= LSE_ATOL
        # and against the float64 oracle on the same values
        f = oracle.forward(h.cpu(), W.cpu(), y.cpu())
        assert abs(loss_s.item() - f["loss"]) <= LOSS_RTOL * abs(f["loss"])
        err = np.max(np.abs(lse_s.cpu().double().numpy() - f["lse"]))
        assert err <= LSE_ATOL


@pytest.mark.parametrize("V", [8192, 7600])
def test_static_forward_at_the_row_limit(V):
    """L = 131072 (the limit) and H = 20480. With V = 8192 (32 column
    tiles) the column-split choice wants 16 splits, more than the 15 whose
    partials fit next to the row data at this L, so the call takes 11
    splits of 3 tiles; with V = 7600 (30 tiles) it takes 15 splits of 2,
    whose partials end 0.5 MB before the end of the array. Both against
    lce_forward (which keeps 16 and 15 splits) and sampled rows against
    the float64 oracle."""
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    lib = lce.load()
    wl = Workload(f"static_limit_{V}", 131072, 20480, V, "bf16", 1.0, 0.01,
                  "uniform", ignore_frac=0.05)
    h, W, y = make_inputs(wl, seed=3, device=dev)
    st, loss_s, lse_s = _static_forward(lib, h, W, y)
    assert st == 0, lib.lce_last_cuda_error().decode()
    assert lce.get_error() == 0
    loss_w, lse_w = lce.forward(h, W, y)
    assert lce.get_error() == 0
    # the same arithmetic per column split; only the merge order differs
    assert abs(loss_s.item() - loss_w.item()) <= 1e-5 * abs(loss_w.item())
    assert (lse_s - lse_w).abs().max().item() <= 1e-4
    rows = np.array([0, 1, 65535, 131071] +
                    list(np.random.default_rng(5).integers(0, wl.L, 8)))
    r = oracle.rows(h.cpu(), W.cpu(), y.cpu(), rows, want_dH=False)
    err = np.max(np.abs(lse_s[torch.from_numpy(rows).to(dev)].cpu().double()
                        .numpy() - r["lse"]))
    assert err <= LSE_ATOL


def test_static_forward_refuses_rows_above_limit():
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    from chunked_lm_head_gemm_gb300 import _binding as B
    lib = lce.load()
    L, H, V = 131073, 8, 16
    h = torch.zeros(L, H, dtype=torch.bfloat16, device=dev)
    W = torch.zeros(V, H, dtype=torch.bfloat16, device=dev)
    y = torch.zeros(L, dtype=torch.int64, device=dev)
    st, _, _ = _static_forward(lib, h, W, y)
    assert st == B.LCE_ERR_WORKSPACE
    assert b"131072" in lib.lce_last_cuda_error()
    assert lce.get_error() == 0
