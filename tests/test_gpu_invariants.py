"""Properties of the loss that hold at any size, checked at full head shape
in the launch configuration the benchmark times, plus a full-length dW
check against the float64 oracle on a reduced vocabulary.

The loss is a sum over rows, each softmax running along one row's
vocabulary ("Training Beyond 1M Tokens", section "The massive logits matrix:
chunk it"). Hence:
  - a common shift of one row's logits (W -> W + 1 u^T adds h_i . u to every
    logit of row i) moves lse by h_i . u and changes neither the loss nor
    dH nor dW (the rows of softmax - onehot sum to zero);
  - permuting the rows permutes lse and dH and leaves the loss and dW
    unchanged;
  - the rows can be cut into chunks at will: at every head shape's full
    length and default chunk, dW (accumulated over all chunks) equals the
    oracle's on every row of a reduced vocabulary.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from chunked_lm_head_gemm_gb300.inputs import WORKLOADS, make_inputs
from tests.gpu_util import (GRAD_RFRO, LOSS_RTOL, LSE_ATOL, MODES, rel_fro,
                            require_gpu, to64)

pytestmark = pytest.mark.gpu


def _run(lce, h, W, y, mode, ws):
    dloss = torch.ones((), device=h.device)
    if mode == "fused":
        loss, lse, dH, dW = lce.forward_backward(h, W, y, workspace=ws)
    else:
        loss, lse = lce.forward(h, W, y, workspace=ws)
        dH, dW = lce.backward(h, W, y, lse, dloss, workspace=ws)
    assert lce.get_error() == 0
    return loss, lse, dH, dW


@pytest.mark.parametrize("mode", MODES)
def test_shift_invariance_full_head(mode):
    """8B head shape, full L. The shift is made exact in bf16: the last 8
    columns of W are zero in problem A and the bf16 constants c in problem
    B, so W_B = W_A + 1 u^T with u = (0, ..., 0, c) and every logit of row
    i moves by exactly s_i = h_i[-8:] . c."""
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    wl = WORKLOADS["qwen3-8b"]
    h, W, y = make_inputs(wl, seed=0, device=dev)
    c = torch.tensor([0.5, -1.0, 0.25, 2.0, -0.75, 1.5, -2.0, 1.0],
                     dtype=torch.bfloat16, device=dev)
    W[:, -8:] = 0
    ws = lce.alloc_workspace(wl.L, wl.H, wl.V, h.dtype, 0, dev)
    loss_a, lse_a, dH_a, dW_a = _run(lce, h, W, y, mode, ws)
    W[:, -8:] = c
    loss_b, lse_b, dH_b, dW_b = _run(lce, h, W, y, mode, ws)
    shift = h[:, -8:].double() @ c.double()
    assert shift.abs().max().item() > 5.0  # a shift that matters
    assert abs(loss_b.item() - loss_a.item()) <= 1e-5 * abs(loss_a.item())
    err = (lse_b.double() - lse_a.double() - shift).abs().max().item()
    assert err <= 1e-4, f"lse moved by h.u +- {err}"
    e = rel_fro(to64(dH_b), to64(dH_a))
    assert e <= GRAD_RFRO / 10, f"dH changed by {e}"
    e = rel_fro(to64(dW_b), to64(dW_a))
    assert e <= GRAD_RFRO / 10, f"dW changed by {e}"


@pytest.mark.parametrize("mode", MODES)
def test_row_permutation_full_head(mode):
    """8B head shape, full L, rows of h and labels permuted. The recomputing
    path computes every row with the same arithmetic wherever it sits, so
    lse and dH permute bit for bit; the fused path's per-chunk column
    splits depend on the chunk's row count (the last chunk is shorter), so
    there they permute up to fp32 rounding. dW differs only in the fp32
    order in which rows of different chunks add up."""
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    wl = WORKLOADS["qwen3-8b"]
    h, W, y = make_inputs(wl, seed=0, device=dev)
    ws = lce.alloc_workspace(wl.L, wl.H, wl.V, h.dtype, 0, dev)
    loss, lse, dH, dW = _run(lce, h, W, y, mode, ws)
    g = torch.Generator(device="cpu").manual_seed(12)
    p = torch.randperm(wl.L, generator=g).to(dev)
    hp, yp = h[p].contiguous(), y[p].contiguous()
    del h
    loss_p, lse_p, dH_p, dW_p = _run(lce, hp, W, yp, mode, ws)
    assert abs(loss_p.item() - loss.item()) <= 1e-6 * abs(loss.item())
    if mode == "separate":
        assert torch.equal(lse_p, lse[p])
        assert torch.equal(dH_p, dH[p])
    else:
        assert (lse_p - lse[p]).abs().max().item() <= 1e-5
        assert rel_fro(to64(dH_p), to64(dH[p])) <= GRAD_RFRO / 10
    e = rel_fro(to64(dW_p), to64(dW))
    bound = 1e-4 if mode == "separate" else GRAD_RFRO / 10
    assert e <= bound, f"dW changed by {e}"


# (head shape, its default backward chunk at the full vocabulary)
FULL_LENGTH = [("qwen3-0.6b", 24320), ("qwen3-4b", 19456),
               ("qwen3-8b", 24320), ("qwen3-32b", 19456)]


@pytest.mark.parametrize("name,chunk", FULL_LENGTH,
                         ids=[f[0] for f in FULL_LENGTH])
def test_full_length_dW_against_oracle(name, chunk):
    """Every row of a head shape's workload (full L and H, its label
    recipe: uniform, Zipf at 4B where the most frequent id takes ~18% of
    the rows, x20 stress rows at 32B) against a reduced vocabulary of 520
    ids (two full 256-column tiles and a ragged one), backward in the
    shape's default row chunks at the full vocabulary (the chunking the
    benchmark runs): dW on every vocabulary row, accumulated over every
    chunk, against the float64 oracle; also the loss, every lse and 64
    sampled dH rows. Both paths, default contraction variant."""
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    wl = dataclasses.replace(WORKLOADS[name], V=520, name=f"{name}-v520")
    h, W, y = make_inputs(wl, seed=0, device=dev)
    L, H, V = wl.L, wl.H, wl.V
    assert L > chunk  # several chunks
    ws = lce.alloc_workspace(L, H, V, h.dtype, chunk, dev)
    ref = oracle.forward_backward(h.cpu(), W.cpu(), y.cpu(), dloss=1.0,
                                  want_dH=False)
    rows = np.unique(np.concatenate(
        [[0, chunk - 1, chunk, L - 1],
         np.random.default_rng(13).integers(0, L, 60)]))
    r = oracle.rows(h.cpu(), W.cpu(), y.cpu(), rows, dloss=1.0)
    dloss = torch.ones((), device=dev)
    for mode in MODES:
        if mode == "fused":
            loss, lse, dH, dW = lce.forward_backward(h, W, y, chunk_rows=chunk,
                                                     workspace=ws)
        else:
            loss, lse = lce.forward(h, W, y, workspace=ws)
            dH, dW = lce.backward(h, W, y, lse, dloss, chunk_rows=chunk,
                                  workspace=ws)
        assert lce.get_error() == 0
        assert abs(loss.item() - ref["loss"]) <= LOSS_RTOL * abs(ref["loss"])
        assert np.max(np.abs(to64(lse) - ref["lse"])) <= LSE_ATOL
        e = rel_fro(to64(dW), ref["dW"])
        assert e <= GRAD_RFRO, f"{mode}: dW rel Frobenius err {e}"
        e = rel_fro(to64(dH[torch.from_numpy(rows).to(dev)]), r["dH"])
        assert e <= GRAD_RFRO, f"{mode}: sampled dH rows err {e}"
