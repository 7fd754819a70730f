"""Label smoothing and z-loss on the GPU against the float64 oracle.

Neither variant is on the pages, which define only the plain cross entropy
("Training Beyond 1M Tokens", section "The loss is the first thing to
break"). The reading: label smoothing eps takes each valid row's cross
entropy against the target (1 - eps) onehot + eps / V; the z-loss adds
coef * lse^2 per valid row; the mean runs over the valid rows. Both paths
(recomputing and fused) and both contraction variants, on the small
workload (fp32 inputs), a ragged multi-tile shape with several backward
chunks, and row slices of the 8B and 32B head shapes (full H and V; the
32B slice with its x20 stress rows). With both
options 0 the _ex calls give the plain calls' bits.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from chunked_lm_head_gemm_gb300.inputs import WORKLOADS, Workload, make_inputs
from tests.gpu_util import (MODES, PAIRS, assert_parity, rel_fro,
                            require_gpu, run_gpu)

pytestmark = pytest.mark.gpu

VARIANTS = [(0.1, 0.0), (0.0, 1e-2), (0.2, 1e-3), (1.0, 0.0)]
CASES = {
    "tiny": (WORKLOADS["tiny"], 0),
    "multi_tile": (Workload("multi_tile", 640, 256, 4100, "bf16", 1.0, 0.05,
                            "uniform", ignore_frac=0.05), 256),
    "qwen3-8b[L=256]": (WORKLOADS["qwen3-8b"].with_rows(256), 0),
    # the widest head, with its x20 stress rows (the largest logits, so the
    # largest lse in the z-loss term)
    "qwen3-32b[L=256]": (WORKLOADS["qwen3-32b"].with_rows(256), 0),
}
_CACHE = {}


def _inputs(case, dev):
    wl, chunk = CASES[case]
    h, W, y = make_inputs(wl, seed=2, device=dev)
    return wl, chunk, h, W, y


def _oracle(case, eps, zc, h, W, y, vrows):
    key = (case, eps, zc)
    if key not in _CACHE:
        fb = oracle.forward_backward(h.cpu(), W.cpu(), y.cpu(), dloss=1.5,
                                     vrows=vrows, label_smoothing=eps,
                                     z_loss=zc)
        _CACHE[key] = fb
    return _CACHE[key]


@pytest.mark.parametrize("pair", PAIRS, ids=lambda v: "pair" if v else "cta")
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("eps,zc", VARIANTS,
                         ids=[f"eps{e}-z{z}" for e, z in VARIANTS])
@pytest.mark.parametrize("case", list(CASES))
def test_variant_parity(case, eps, zc, mode, pair):
    dev = require_gpu()
    wl, chunk, h, W, y = _inputs(case, dev)
    gpu = run_gpu(h, W, y, dloss=1.5, chunk_rows=chunk, mode=mode, pair=pair,
                  label_smoothing=eps, z_loss=zc)
    assert gpu["status"] == 0
    vrows = None
    if wl.V > 10000:
        yc = y.cpu().numpy()
        rs = np.random.default_rng(7)
        vrows = np.unique(np.concatenate(
            [yc[yc >= 0], rs.integers(0, wl.V, 256), [0, wl.V - 1]]))
    fb = _oracle(case, eps, zc, h, W, y, vrows)
    assert_parity(gpu, fb, fb, dW_rows=vrows)


@pytest.mark.parametrize("mode", MODES)
def test_zero_options_are_the_plain_call(mode):
    """lce_*_ex with {0, 0} runs the plain arithmetic: identical bits."""
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    from chunked_lm_head_gemm_gb300 import _binding as B
    lib = lce.load()
    wl, chunk, h, W, y = _inputs("multi_tile", dev)
    L, H = h.shape
    V = W.shape[0]
    ws = lce.alloc_workspace(L, H, V, h.dtype, chunk, dev)
    s = torch.cuda.current_stream().cuda_stream
    zero = ctypes.pointer(B.LossOpts(0.0, 0.0))
    loss = torch.empty((), dtype=torch.float32, device=dev)
    lse = torch.empty(L, dtype=torch.float32, device=dev)
    dH = torch.empty_like(h)
    dW = torch.empty(V, H, dtype=torch.float32, device=dev)
    one = torch.ones(1, device=dev)
    if mode == "fused":
        st = lib.lce_forward_backward_ex(
            h.data_ptr(), W.data_ptr(), 0, y.data_ptr(), L, H, V, -100, zero,
            chunk, loss.data_ptr(), lse.data_ptr(), dH.data_ptr(),
            dW.data_ptr(), ws.data_ptr(), ws.numel(), s)
        assert st == 0
        ref = lce.forward_backward(h, W, y, chunk_rows=chunk, workspace=ws)
    else:
        st = lib.lce_forward_ex(h.data_ptr(), W.data_ptr(), 0, y.data_ptr(),
                                L, H, V, -100, zero, loss.data_ptr(),
                                lse.data_ptr(), ws.data_ptr(), ws.numel(), s)
        assert st == 0
        st = lib.lce_backward_ex(h.data_ptr(), W.data_ptr(), 0, y.data_ptr(),
                                 lse.data_ptr(), L, H, V, -100, zero,
                                 one.data_ptr(), chunk, dH.data_ptr(),
                                 dW.data_ptr(), ws.data_ptr(), ws.numel(), s)
        assert st == 0
        rl, rlse = lce.forward(h, W, y, workspace=ws)
        rdH, rdW = lce.backward(h, W, y, rlse, one, chunk_rows=chunk,
                                workspace=ws)
        ref = (rl, rlse, rdH, rdW)
    assert lce.get_error() == 0
    for a, b in zip((loss, lse, dH, dW), ref):
        assert torch.equal(a, b)


@pytest.mark.parametrize("mode", MODES)
def test_variant_autograd(mode):
    """linear_cross_entropy with both options: the same loss and gradients
    as the explicit calls, and the oracle's."""
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    wl, chunk, h, W, y = _inputs("multi_tile", dev)
    kw = dict(label_smoothing=0.2, z_loss=1e-3)
    hh = h.clone().requires_grad_(True)
    WW = W.clone().requires_grad_(True)
    loss = lce.linear_cross_entropy(hh, WW, y, chunk_rows=chunk,
                                    fused=(mode == "fused"), **kw)
    (1.5 * loss).backward()
    gpu = run_gpu(h, W, y, dloss=1.5, chunk_rows=chunk, mode=mode, **kw)
    assert loss.item() == gpu["loss"]
    assert torch.equal(hh.grad.float().cpu(),
                       torch.from_numpy(gpu["dH"]).float())
    fb = _oracle("multi_tile", 0.2, 1e-3, h, W, y, None)
    assert rel_fro(WW.grad.double().cpu().numpy(), fb["dW"]) < 1e-2


def test_variants_full_size_sampled_rows():
    """The 8B shard at full size with label smoothing and the z-loss, in the
    launch configuration the benchmark times (fused path, default chunk):
    lse and dH on sampled rows (first, last, an ignored one, random)
    against the oracle's rows of the whole problem (its N over all
    labels); the loss against its definition given lse over every row; the
    recomputing path within the bound of the fused one."""
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    from tests.gpu_util import GRAD_RFRO, LSE_ATOL, to64
    wl = WORKLOADS["qwen3-8b"]
    h, W, y = make_inputs(wl, seed=0, device=dev)
    kw = dict(label_smoothing=0.1, z_loss=1e-4)
    ws = lce.alloc_workspace(wl.L, wl.H, wl.V, h.dtype, 0, dev)
    loss, lse, dH, dW = lce.forward_backward(h, W, y, workspace=ws, **kw)
    assert lce.get_error() == 0
    rs = np.random.default_rng(17)
    rows = np.unique(np.concatenate([[0, wl.L - 1],
                                     rs.integers(0, wl.L, 10)]))
    r = oracle.rows(h.cpu(), W.cpu(), y.cpu(), rows, dloss=1.0, **kw)
    idx = torch.from_numpy(rows).to(dev)
    assert np.max(np.abs(to64(lse)[rows] - r["lse"])) <= LSE_ATOL
    e = rel_fro(to64(dH[idx]), r["dH"])
    assert e <= GRAD_RFRO, f"sampled dH rows rel Frobenius err {e}"
    # the loss from its definition given lse, every row: the mean over
    # valid rows of lse - (1 - eps) z_y - (eps / V) sum_j z_j + coef lse^2,
    # with z_y = h_i . W_y and sum_j z_j = h_i . (sum_j W_j) in float64
    eps, zc = kw["label_smoothing"], kw["z_loss"]
    valid = (y >= 0) & (y < wl.V)
    idx_v = torch.nonzero(valid).flatten()
    zy = torch.zeros(wl.L, dtype=torch.float64, device=dev)
    for s0 in range(0, idx_v.numel(), 8192):
        ii = idx_v[s0:s0 + 8192]
        zy[ii] = (h[ii].double() * W[y[ii]].double()).sum(1)
    wsum = W.double().sum(0)
    zsum = torch.cat([h[r0:r0 + 8192].double() @ wsum
                      for r0 in range(0, wl.L, 8192)])
    l64 = lse.double()
    term = l64 - (1 - eps) * zy - eps / wl.V * zsum + zc * l64 ** 2
    ref_loss = term[valid].mean().item()
    assert abs(loss.item() - ref_loss) <= 1e-4 * abs(ref_loss)
    # and plausible against the plain loss: plus the z-loss term, minus at
    # most eps times the spread of the logits
    plain, _ = lce.forward(h, W, y, workspace=ws)
    zl = zc * (l64[valid] ** 2).mean().item()
    assert abs(loss.item() - (plain.item() + zl)) < 0.1 * plain.item()
    # the recomputing path agrees with the fused one
    one = torch.ones((), device=dev)
    loss2, lse2 = lce.forward(h, W, y, workspace=ws, **kw)
    dH2, dW2 = lce.backward(h, W, y, lse2, one, workspace=ws, **kw)
    assert lce.get_error() == 0
    assert abs(loss2.item() - loss.item()) <= 1e-5 * abs(loss.item())
    assert rel_fro(to64(dH2), to64(dH)) <= GRAD_RFRO
    assert rel_fro(to64(dW2), to64(dW)) <= GRAD_RFRO


@pytest.mark.parametrize("mode", MODES)
def test_variant_edge_cases(mode):
    """Loss variants on the degenerate cases: every row ignored (loss 0,
    gradients 0), one class (smoothing changes nothing, the z-loss
    remains), labels out of range (reported and ignored)."""
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300._binding as B
    kw = dict(label_smoothing=0.3, z_loss=0.02)
    wl = Workload("vallign", 150, 32, 400, "bf16", 1.0, 0.1, "uniform")
    h, W, y = make_inputs(wl, seed=3, device=dev)
    y[:] = -100
    gpu = run_gpu(h, W, y, mode=mode, **kw)
    assert gpu["status"] == 0 and gpu["loss"] == 0.0
    assert np.all(gpu["dH"] == 0.0) and np.all(gpu["dW"] == 0.0)
    for name, L, H, V, seed in (("v1", 70, 16, 1, 2), ("vbad", 260, 32, 500, 4)):
        wl = Workload(name, L, H, V, "bf16", 1.0, 0.5 if V == 1 else 0.1,
                      "uniform", ignore_frac=0.1)
        h, W, y = make_inputs(wl, seed=seed, device=dev)
        if name == "vbad":
            y[3] = 500
            y[77] = -7
        gpu = run_gpu(h, W, y, dloss=0.8, mode=mode, **kw)
        fb = oracle.forward_backward(h.cpu(), W.cpu(), y.cpu(), dloss=0.8,
                                     **kw)
        if name == "vbad":
            assert gpu["status"] == B.LCE_ERR_LABEL_RANGE
            assert fb["status"] == oracle.LABEL_RANGE
        else:
            assert gpu["status"] == 0
        assert_parity(gpu, fb, fb)
