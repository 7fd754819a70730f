"""The sequence-tiled gated MLP on the GPU against its float64 oracle:
y = (silu(x Wg^T) * (x Wu^T)) Wd^T and its backward, over row chunks, on
single-CTA and CTA-pair contractions."""
import numpy as np
import pytest
import torch

import oracle
from chunked_lm_head_gemm_gb300.inputs import (MLP_WORKLOADS, MlpWorkload,
                                               make_mlp_inputs)
from tests.gpu_util import PAIRS, cta_pair, rel_fro, require_gpu, to64

pytestmark = pytest.mark.gpu

TOL = 1e-2  # relative Frobenius error, bf16 operands and intermediates


def _run(x, Wg, Wu, Wd, dy, chunk):
    import chunked_lm_head_gemm_gb300 as lce
    y = lce.mlp_forward(x, Wg, Wu, Wd, chunk)
    dx, dWg, dWu, dWd = lce.mlp_backward(x, Wg, Wu, Wd, dy, chunk)
    assert lce.get_error() == 0
    return dict(y=to64(y), dx=to64(dx), dWg=to64(dWg), dWu=to64(dWu),
                dWd=to64(dWd))


def _compare(gpu, ref):
    for k in ("y", "dx", "dWg", "dWu", "dWd"):
        e = rel_fro(gpu[k], ref[k])
        assert e <= TOL, f"{k} rel Frobenius err {e}"


SHAPES = [
    # name, L, H, I, chunk, x_scale, w_std
    ("tiny", 200, 64, 128, 0, 1.0, 0.1),
    ("ragged", 333, 136, 192, 128, 1.0, 0.1),
    ("one_row", 1, 8, 64, 0, 1.0, 0.3),
    ("chunk_100", 300, 256, 320, 100, 1.0, 0.05),
    ("multi_tile", 700, 512, 1024, 256, 1.0, 0.03),
]


@pytest.mark.parametrize("pair", PAIRS, ids=lambda v: "pair" if v else "cta")
@pytest.mark.parametrize("name,L,H,I,chunk,xs,ws", SHAPES,
                         ids=[s_[0] for s_ in SHAPES])
def test_mlp_against_oracle(name, L, H, I, chunk, xs, ws, pair):
    dev = require_gpu()
    wl = MlpWorkload(name, L, H, I, xs, ws)
    x, Wg, Wu, Wd, dy = make_mlp_inputs(wl, seed=1, device=dev)
    with cta_pair(pair):
        gpu = _run(x, Wg, Wu, Wd, dy, chunk)
    ref = oracle.mlp(x.cpu(), Wg.cpu(), Wu.cpu(), Wd.cpu(), dy.cpu())
    _compare(gpu, ref)


@pytest.mark.parametrize("pair", PAIRS, ids=lambda v: "pair" if v else "cta")
@pytest.mark.parametrize("name", ["qwen3-0.6b-mlp", "qwen3-4b-mlp",
                                  "qwen3-8b-mlp", "qwen3-32b-mlp"])
def test_mlp_row_slice_of_qwen3_shape(name, pair):
    """256 rows at the Qwen3 MLP widths (H, I), the oracle on all of it."""
    dev = require_gpu()
    wl = MLP_WORKLOADS[name].with_rows(256)
    x, Wg, Wu, Wd, dy = make_mlp_inputs(wl, seed=0, device=dev)
    with cta_pair(pair):
        gpu = _run(x, Wg, Wu, Wd, dy, 0)
    ref = oracle.mlp(x.cpu(), Wg.cpu(), Wu.cpu(), Wd.cpu(), dy.cpu())
    _compare(gpu, ref)


def test_mlp_multichunk_slice_of_qwen3_8b():
    """1024 rows at the Qwen3-8B MLP widths in 256-row chunks: the weight
    gradients' fp32 read-add-write runs three times at full H and I, the
    intermediates are recomputed per chunk; all five outputs against the
    oracle."""
    dev = require_gpu()
    wl = MLP_WORKLOADS["qwen3-8b-mlp"].with_rows(1024)
    x, Wg, Wu, Wd, dy = make_mlp_inputs(wl, seed=2, device=dev)
    gpu = _run(x, Wg, Wu, Wd, dy, 256)
    ref = oracle.mlp(x.cpu(), Wg.cpu(), Wu.cpu(), Wd.cpu(), dy.cpu())
    _compare(gpu, ref)


def test_mlp_chunking_and_determinism():
    """Rows do not depend on the chunking (y, dx bitwise); weight gradients
    only through fp32 summation order; reruns are bitwise identical."""
    dev = require_gpu()
    wl = MlpWorkload("det", 1536, 256, 512, 1.0, 0.05)
    x, Wg, Wu, Wd, dy = make_mlp_inputs(wl, seed=3, device=dev)
    a = _run(x, Wg, Wu, Wd, dy, 0)
    b = _run(x, Wg, Wu, Wd, dy, 0)
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    c = _run(x, Wg, Wu, Wd, dy, 512)
    assert np.array_equal(a["y"], c["y"]) and np.array_equal(a["dx"], c["dx"])
    for k in ("dWg", "dWu", "dWd"):
        assert rel_fro(c[k], a[k]) < 1e-5, k


def test_mlp_bad_arguments():
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    from chunked_lm_head_gemm_gb300 import _binding as B
    wl = MlpWorkload("bad", 64, 64, 96, 1.0, 0.1)  # I not a multiple of 64
    x, Wg, Wu, Wd, dy = make_mlp_inputs(wl, seed=0, device=dev)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    with pytest.raises(lce.LCEError) as ei:
        lce.mlp_forward(x, Wg, Wu, Wd, workspace=ws)
    assert ei.value.status == B.LCE_ERR_INVALID_ARG
    assert lce.get_error() == 0


def test_mlp_autograd_function():
    """sequence_tiled_mlp under autograd: y, and the gradients of
    sum(y * dy) for x and the three weights, equal the explicit calls'
    bits (dy reaches the backward as the upstream gradient); a second
    backward through a retained graph gives the same; and the oracle
    agrees within the tolerance."""
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    wl = MlpWorkload("ag", 300, 128, 256, 1.0, 0.05)
    x, Wg, Wu, Wd, dy = make_mlp_inputs(wl, seed=8, device=dev)
    leaves = [t.clone().requires_grad_(True) for t in (x, Wg, Wu, Wd)]
    y = lce.sequence_tiled_mlp(*leaves, chunk_rows=128)
    y.backward(dy, retain_graph=True)
    grads = [t.grad.clone() for t in leaves]
    assert all(g.dtype == torch.bfloat16 for g in grads)
    y_ref = lce.mlp_forward(x, Wg, Wu, Wd, 128)
    dx, dWg, dWu, dWd = lce.mlp_backward(x, Wg, Wu, Wd, dy, 128)
    assert lce.get_error() == 0
    assert torch.equal(y.detach(), y_ref)
    for got, want in zip(grads, (dx, dWg.bfloat16(), dWu.bfloat16(),
                                 dWd.bfloat16())):
        assert torch.equal(got, want)
    for t in leaves:
        t.grad = None
    y.backward(dy)
    for t, g in zip(leaves, grads):
        assert torch.equal(t.grad, g)
    ref = oracle.mlp(x.cpu(), Wg.cpu(), Wu.cpu(), Wd.cpu(), dy.cpu())
    got = dict(y=to64(y), dx=to64(grads[0]), dWg=to64(grads[1]),
               dWu=to64(grads[2]), dWd=to64(grads[3]))
    _compare(got, ref)


def test_mlp_optional_gradients():
    """Frozen weights (adapter fine-tuning): dx alone skips the three
    weight-gradient contractions and keeps the full call's bits; the weight
    gradients alone, and dWd alone, likewise; under autograd with the
    weights frozen, x.grad is the full call's dx."""
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    wl = MlpWorkload("opt", 400, 128, 256, 1.0, 0.05)
    x, Wg, Wu, Wd, dy = make_mlp_inputs(wl, seed=11, device=dev)
    full = lce.mlp_backward(x, Wg, Wu, Wd, dy, 128)
    only_dx = lce.mlp_backward(x, Wg, Wu, Wd, dy, 128, compute_dWgu=False,
                               compute_dWd=False)
    assert only_dx[1] is None and only_dx[3] is None
    assert torch.equal(only_dx[0], full[0])
    only_w = lce.mlp_backward(x, Wg, Wu, Wd, dy, 128, compute_dx=False)
    assert only_w[0] is None
    for a, b in zip(only_w[1:], full[1:]):
        assert torch.equal(a, b)
    only_wd = lce.mlp_backward(x, Wg, Wu, Wd, dy, 128, compute_dx=False,
                               compute_dWgu=False)
    assert torch.equal(only_wd[3], full[3])
    with pytest.raises(lce.LCEError):
        lce.mlp_backward(x, Wg, Wu, Wd, dy, 128, compute_dx=False,
                         compute_dWgu=False, compute_dWd=False)
    xx = x.clone().requires_grad_(True)
    y = lce.sequence_tiled_mlp(xx, Wg, Wu, Wd, chunk_rows=128)
    y.backward(dy)
    assert torch.equal(xx.grad, full[0])
    assert lce.get_error() == 0
