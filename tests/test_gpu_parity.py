"""CUDA path against the float64 oracle, element by element, on seeded
inputs small enough for the oracle: the small workload, edge cases, and row
slices (full H and V) of every Qwen3 head shape."""
import numpy as np
import pytest
import torch

import oracle
from chunked_lm_head_gemm_gb300.inputs import (WORKLOADS, Workload,
                                               make_inputs)
from tests.gpu_util import (MODES, PAIRS, assert_parity, rel_fro,
                            require_gpu, run_gpu, to64)

pytestmark = pytest.mark.gpu


def _oracle(h, W, y, dloss=1.0, vrows=None):
    hc, Wc, yc = h.cpu(), W.cpu(), y.cpu()
    f = oracle.forward(hc, Wc, yc)
    b = oracle.backward(hc, Wc, yc, dloss=dloss, vrows=vrows)
    return f, b


# oracle results of the row slices, shared by the parametrisations of one
# slice (both paths, both contraction variants run on the same inputs)
_SLICE_CACHE = {}


def _slice_oracle(key, h, W, y, vrows):
    if key not in _SLICE_CACHE:
        fb = oracle.forward_backward(h.cpu(), W.cpu(), y.cpu(), dloss=1.0,
                                     vrows=vrows)
        _SLICE_CACHE[key] = (fb, fb)
    return _SLICE_CACHE[key]


@pytest.mark.parametrize("pair", PAIRS, ids=lambda v: "pair" if v else "cta")
@pytest.mark.parametrize("mode", MODES)
def test_tiny_workload(mode, pair):
    """512 x 256 x 4096, fp32 inputs, 10% ignored."""
    dev = require_gpu()
    h, W, y = make_inputs("tiny", seed=0, device=dev)
    gpu = run_gpu(h, W, y, mode=mode, pair=pair)
    assert gpu["status"] == 0
    f, b = _oracle(h, W, y)
    assert_parity(gpu, f, b)


EDGE = [
    # name, L, H, V, dtype, chunk_rows, ignore_frac, w_std
    ("ragged_small", 3, 16, 5, "bf16", 0, 0.0, 0.5),
    ("k_below_tile_v_odd", 130, 8, 300, "bf16", 0, 0.1, 0.3),
    ("ragged_k", 257, 72, 1000, "bf16", 0, 0.1, 0.1),
    ("chunk_64", 300, 64, 520, "bf16", 64, 0.1, 0.1),
    ("chunk_100", 300, 64, 520, "bf16", 100, 0.1, 0.1),
    ("multi_tile", 640, 256, 4100, "bf16", 256, 0.05, 0.05),
    ("f32_ragged", 200, 40, 777, "f32", 96, 0.1, 0.1),
    ("one_row", 1, 8, 700, "bf16", 0, 0.0, 0.5),
]


@pytest.mark.parametrize("pair", PAIRS, ids=lambda v: "pair" if v else "cta")
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name,L,H,V,dt,chunk,ign,wstd", EDGE,
                         ids=[e[0] for e in EDGE])
def test_edge_shapes(name, L, H, V, dt, chunk, ign, wstd, mode, pair):
    dev = require_gpu()
    wl = Workload(name, L, H, V, dt, 1.0, wstd, "uniform", ignore_frac=ign)
    h, W, y = make_inputs(wl, seed=1, device=dev)
    gpu = run_gpu(h, W, y, dloss=1.0, chunk_rows=chunk, mode=mode, pair=pair)
    assert gpu["status"] == 0
    f, b = _oracle(h, W, y)
    assert_parity(gpu, f, b)


@pytest.mark.parametrize("mode", MODES)
def test_single_class_gives_zero(mode):
    """V = 1: every lse equals the one logit; loss and gradients vanish."""
    dev = require_gpu()
    wl = Workload("v1", 70, 16, 1, "bf16", 1.0, 0.5, "uniform")
    h, W, y = make_inputs(wl, seed=2, device=dev)
    gpu = run_gpu(h, W, y, mode=mode)
    z = (h.double() @ W.double().T)[:, 0].cpu().numpy()
    assert np.max(np.abs(gpu["lse"] - z)) < 1e-4 * max(1.0, np.max(np.abs(z)))
    assert abs(gpu["loss"]) < 1e-5
    assert np.max(np.abs(gpu["dH"])) < 1e-6 and np.max(np.abs(gpu["dW"])) < 1e-6


@pytest.mark.parametrize("mode", MODES)
def test_all_rows_ignored(mode):
    dev = require_gpu()
    wl = Workload("allign", 150, 32, 400, "bf16", 1.0, 0.1, "uniform")
    h, W, y = make_inputs(wl, seed=3, device=dev)
    y[:] = -100
    gpu = run_gpu(h, W, y, mode=mode)
    assert gpu["status"] == 0
    assert gpu["loss"] == 0.0
    assert np.all(gpu["dH"] == 0.0) and np.all(gpu["dW"] == 0.0)
    f = oracle.forward(h.cpu(), W.cpu(), y.cpu())
    assert np.max(np.abs(gpu["lse"] - f["lse"])) < 2e-3


@pytest.mark.parametrize("mode", MODES)
def test_labels_out_of_range_are_reported_and_ignored(mode):
    dev = require_gpu()
    wl = Workload("bad", 260, 32, 500, "bf16", 1.0, 0.1, "uniform",
                  ignore_frac=0.1)
    h, W, y = make_inputs(wl, seed=4, device=dev)
    y[3] = 500
    y[77] = -7
    y[200] = 10 ** 12
    gpu = run_gpu(h, W, y, mode=mode)
    import chunked_lm_head_gemm_gb300._binding as B
    assert gpu["status"] == B.LCE_ERR_LABEL_RANGE
    f, b = _oracle(h, W, y)
    assert f["status"] == oracle.LABEL_RANGE
    assert_parity(gpu, f, b)
    assert B.get_error() == 0  # cleared by the read


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("dloss", [0.0, 2.5, -0.75])
def test_dloss_scaling(dloss, mode):
    dev = require_gpu()
    wl = Workload("dl", 200, 64, 700, "bf16", 1.0, 0.1, "uniform",
                  ignore_frac=0.1)
    h, W, y = make_inputs(wl, seed=5, device=dev)
    gpu = run_gpu(h, W, y, dloss=dloss, mode=mode)
    if dloss == 0.0:
        assert np.all(gpu["dH"] == 0.0) and np.all(gpu["dW"] == 0.0)
        return
    f, b = _oracle(h, W, y, dloss=dloss)
    assert_parity(gpu, f, b)


@pytest.mark.parametrize("mode", MODES)
def test_autograd_function_matches_explicit_calls(mode):
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    wl = Workload("ag", 300, 64, 900, "bf16", 1.0, 0.1, "uniform",
                  ignore_frac=0.1)
    h, W, y = make_inputs(wl, seed=6, device=dev)
    hh = h.clone().requires_grad_(True)
    WW = W.clone().requires_grad_(True)
    loss = lce.linear_cross_entropy(hh, WW, y, fused=(mode == "fused"))
    (3.0 * loss).backward()
    gpu = run_gpu(h, W, y, dloss=3.0, mode=mode)
    assert loss.item() == gpu["loss"]
    assert torch.equal(hh.grad.float().cpu(),
                       torch.from_numpy(gpu["dH"]).float())
    assert rel_fro(WW.grad.double().cpu().numpy(), gpu["dW"]) < 4e-3


@pytest.mark.parametrize("mode", MODES)
def test_autograd_backward_twice(mode):
    """A retained graph can be differentiated again with the same result:
    the fused mode scales copies of the gradients it keeps, never the kept
    tensors themselves, so a second backward (or a non-unit upstream
    gradient) does not scale them twice."""
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    wl = Workload("ag2", 260, 64, 700, "bf16", 1.0, 0.1, "uniform",
                  ignore_frac=0.1)
    h, W, y = make_inputs(wl, seed=8, device=dev)
    hh = h.clone().requires_grad_(True)
    WW = W.clone().requires_grad_(True)
    loss = lce.linear_cross_entropy(hh, WW, y, fused=(mode == "fused"))
    (2.5 * loss).backward(retain_graph=True)
    gh, gw = hh.grad.clone(), WW.grad.clone()
    hh.grad = None
    WW.grad = None
    (2.5 * loss).backward(retain_graph=True)
    assert torch.equal(hh.grad, gh) and torch.equal(WW.grad, gw)
    (2.5 * loss).backward()  # accumulates onto the second pass's gradients
    assert torch.equal(hh.grad, 2 * gh) and torch.equal(WW.grad, 2 * gw)
    gpu = run_gpu(h, W, y, dloss=2.5, mode=mode)
    assert torch.equal(gh.float().cpu(), torch.from_numpy(gpu["dH"]).float())


SLICES = [("qwen3-0.6b", 256), ("qwen3-4b", 300), ("qwen3-8b", 256),
          ("qwen3-32b", 256)]


@pytest.mark.parametrize("pair", PAIRS, ids=lambda v: "pair" if v else "cta")
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name,rows", SLICES, ids=[s[0] for s in SLICES])
def test_row_slice_of_head_shape(name, rows, mode, pair):
    """The first rows of each head shape (full H and V = 151936); dW is
    compared on the vocabulary rows the slice's labels touch, plus 256
    seeded others and the last id."""
    dev = require_gpu()
    wl = WORKLOADS[name].with_rows(rows)
    h, W, y = make_inputs(wl, seed=0, device=dev)
    gpu = run_gpu(h, W, y, dloss=1.0, mode=mode, pair=pair)
    assert gpu["status"] == 0
    vrows = _touched_vocab_rows(y, wl.V)
    f, b = _slice_oracle((name, rows), h, W, y, vrows)
    assert_parity(gpu, f, b, dW_rows=vrows)


def _touched_vocab_rows(y, V):
    """The vocabulary rows the labels touch, 256 seeded others, 0 and V-1."""
    yc = y.cpu().numpy()
    rs = np.random.default_rng(7)
    return np.unique(np.concatenate([yc[yc >= 0], rs.integers(0, V, 256),
                                     [0, V - 1]]))


MULTI = [("qwen3-8b", 1024), ("qwen3-32b", 1024)]


@pytest.mark.parametrize("pair", PAIRS, ids=lambda v: "pair" if v else "cta")
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name,rows", MULTI, ids=[s[0] for s in MULTI])
def test_multichunk_row_slice_of_head_shape(name, rows, mode, pair):
    """1024 rows of the 8B and 32B head shapes (full H and V = 151936; the
    32B slice holds stress rows scaled x20) with a 256-row backward chunk:
    four chunks, so dW's fp32 read-add-write runs three times at full H and
    V, and the fused path writes its tile exponentials four times. Loss,
    every lse, every dH row, and dW on the touched vocabulary rows plus 256
    seeded others and V-1, against the float64 oracle. The loss is a sum
    over rows ("Training Beyond 1M Tokens", section "The massive logits
    matrix: chunk it"), so any chunking must give the oracle's answer."""
    dev = require_gpu()
    wl = WORKLOADS[name].with_rows(rows)
    h, W, y = make_inputs(wl, seed=0, device=dev)
    gpu = run_gpu(h, W, y, dloss=1.0, chunk_rows=256, mode=mode, pair=pair)
    assert gpu["status"] == 0
    vrows = _touched_vocab_rows(y, wl.V)
    f, b = _slice_oracle((name, rows), h, W, y, vrows)
    assert_parity(gpu, f, b, dW_rows=vrows)


@pytest.mark.parametrize("mode", MODES)
def test_optional_gradients(mode):
    """Skipping dW (a frozen head) or dH skips that contraction and leaves
    the other gradient, the loss and lse with the full call's bits; with
    neither, the fused call still gives the loss and lse, and the
    recomputing backward refuses the call."""
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    wl = Workload("optional", 640, 128, 4100, "bf16", 1.0, 0.05, "uniform",
                  ignore_frac=0.1)
    h, W, y = make_inputs(wl, seed=9, device=dev)
    d = torch.full((), 0.5, device=dev)

    def run(cdh, cdw):
        if mode == "fused":
            loss, lse, dH, dW = lce.forward_backward(
                h, W, y, chunk_rows=256, compute_dH=cdh, compute_dW=cdw)
            lce.scale_gradients(dH, dW, d)
        else:
            loss, lse = lce.forward(h, W, y)
            dH, dW = lce.backward(h, W, y, lse, d, chunk_rows=256,
                                  compute_dH=cdh, compute_dW=cdw)
        return loss, lse, dH, dW

    full = run(True, True)
    only_dH = run(True, False)
    only_dW = run(False, True)
    assert only_dH[3] is None and only_dW[2] is None
    assert torch.equal(only_dH[2], full[2])
    assert torch.equal(only_dW[3], full[3])
    for part in (only_dH, only_dW):
        assert torch.equal(part[0], full[0]) and torch.equal(part[1], full[1])
    if mode == "fused":
        loss, lse, dH, dW = lce.forward_backward(h, W, y, chunk_rows=256,
                                                 compute_dH=False,
                                                 compute_dW=False)
        assert dH is None and dW is None
        assert torch.equal(loss, full[0]) and torch.equal(lse, full[1])
    else:
        with pytest.raises(lce.LCEError):
            lce.backward(h, W, y, full[1], d, compute_dH=False,
                         compute_dW=False)
    assert lce.get_error() == 0
    f, b = _oracle(h, W, y, dloss=0.5)
    gpu = dict(loss=full[0].item(), lse=to64(full[1]), dH=to64(only_dH[2]),
               dW=to64(only_dW[3]), status=0)
    assert_parity(gpu, f, b)


@pytest.mark.parametrize("fused", [False, True], ids=["recompute", "fused"])
def test_autograd_frozen_head_or_input(fused):
    """The autograd Function computes only the gradients autograd asks for:
    a frozen head (W without grad) gives h.grad with the bits of the full
    call's dH and no W.grad; a frozen input the converse."""
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    wl = Workload("frozen", 300, 64, 900, "bf16", 1.0, 0.1, "uniform",
                  ignore_frac=0.1)
    h, W, y = make_inputs(wl, seed=10, device=dev)
    one = torch.ones((), device=dev)
    if fused:
        _, _, dH, dW = lce.forward_backward(h, W, y)
    else:
        _, lse = lce.forward(h, W, y)
        dH, dW = lce.backward(h, W, y, lse, one)
    hh = h.clone().requires_grad_(True)
    loss = lce.linear_cross_entropy(hh, W, y, fused=fused)
    loss.backward()
    assert torch.equal(hh.grad, dH)
    WW = W.clone().requires_grad_(True)
    loss = lce.linear_cross_entropy(h, WW, y, fused=fused)
    loss.backward()
    assert torch.equal(WW.grad, dW.to(W.dtype))
    assert lce.get_error() == 0
