"""Vocabulary-parallel form on one GPU, the slices run one after another:
each slice's statistics against the float64 oracle applied to that slice's
sub-vocabulary, the merged lse and loss against the oracle on the whole
vocabulary, and the slices' backward (sum of dH partials, concatenated dW)
against the oracle's gradients."""
import numpy as np
import pytest
import torch

import oracle
import chunked_lm_head_gemm_gb300 as lce
from chunked_lm_head_gemm_gb300 import _binding as B
from chunked_lm_head_gemm_gb300 import vocab_parallel as vp
from chunked_lm_head_gemm_gb300.inputs import Workload, make_inputs
from tests.gpu_util import (GRAD_RFRO, LOSS_RTOL, LSE_ATOL, PAIRS, cta_pair,
                            rel_fro, require_gpu, to64)

pytestmark = pytest.mark.gpu

CASES = [
    # name, L, H, V, slice sizes, chunk_rows
    ("three_ragged", 300, 64, 1000, [333, 333, 334], 0),
    ("four_even", 513, 128, 4096, [1024] * 4, 256),
    ("uneven_tiny_slice", 200, 40, 777, [700, 70, 7], 96),
]


def _bounds(sizes):
    out, v0 = [], 0
    for n in sizes:
        out.append((v0, n))
        v0 += n
    return out


def _slice_oracle(h, Ws, y, v0, Vs):
    """The oracle's forward on the sub-vocabulary: labels in the slice
    mapped to local ids, the rest ignored (they add no label logit)."""
    y = y.clone()
    local = (y >= v0) & (y < v0 + Vs)
    y[~local] = -100
    y[local] -= v0
    return oracle.forward(h, Ws, y), local.numpy()


def _inputs(name, L, H, V, seed=11):
    wl = Workload(name, L, H, V, "bf16", 1.0, 0.1, "uniform", ignore_frac=0.1)
    return make_inputs(wl, seed=seed, device=require_gpu())


@pytest.mark.parametrize("keep", [False, True], ids=["recompute", "keep_exp"])
@pytest.mark.parametrize("pair", PAIRS, ids=lambda v: "pair" if v else "cta")
@pytest.mark.parametrize("name,L,H,V,sizes,chunk", CASES,
                         ids=[c[0] for c in CASES])
def test_slices_forward_backward(name, L, H, V, sizes, chunk, pair, keep):
    h, W, y = _inputs(name, L, H, V)
    hc, Wc, yc = h.cpu(), W.cpu(), y.cpu()
    dloss = torch.full((), 0.5, device=h.device)
    # keep: each slice keeps its exponentials in its own workspace
    wss = [B.slice_exp_workspace(L, H, Vs, h.dtype, h.device) if keep
           else None for _, Vs in _bounds(sizes)]
    with cta_pair(pair):
        stats = []
        for k, (v0, Vs) in enumerate(_bounds(sizes)):
            if keep:
                m, s, zy = B.forward_slice_exp(h, W[v0:v0 + Vs], y, v0, V,
                                               wss[k])
            else:
                m, s, zy = B.forward_slice(h, W[v0:v0 + Vs], y, v0, V)
            stats.append(torch.stack([m, s, zy]))
            # the slice's own statistics against the oracle on its columns
            f_s, local = _slice_oracle(hc, Wc[v0:v0 + Vs], yc, v0, Vs)
            lse_s = (m.double() + torch.log(s.double())).cpu().numpy()
            assert np.max(np.abs(lse_s - f_s["lse"])) <= LSE_ATOL
            zy_h = zy.cpu().numpy()
            assert np.all(zy_h[~local] == 0.0)
            assert np.max(np.abs(zy_h[local] - f_s["zy"][local]),
                          initial=0.0) <= LSE_ATOL
        allst = torch.stack(stats)
        loss, lse = B.combine_slices(allst[:, 0].contiguous(),
                                     allst[:, 1].contiguous(),
                                     allst[:, 2].contiguous(), y, V)
        dH = torch.zeros(L, H, dtype=torch.float32, device=h.device)
        dWs = []
        for k, (v0, Vs) in enumerate(_bounds(sizes)):
            if keep:
                dH_part, dW_s = B.backward_slice_exp(h, W[v0:v0 + Vs], y, lse,
                                                     dloss, v0, V, wss[k])
            else:
                dH_part, dW_s = B.backward_slice(h, W[v0:v0 + Vs], y, lse,
                                                 dloss, v0, V,
                                                 chunk_rows=chunk)
            dH += dH_part
            dWs.append(dW_s)
        dW = torch.cat(dWs)
        assert lce.get_error() == 0
    f = oracle.forward(hc, Wc, yc)
    b = oracle.backward(hc, Wc, yc, dloss=0.5)
    assert abs(loss.item() - f["loss"]) <= LOSS_RTOL * abs(f["loss"])
    assert np.max(np.abs(to64(lse) - f["lse"])) <= LSE_ATOL
    assert rel_fro(to64(dH), b["dH"]) <= GRAD_RFRO
    assert rel_fro(to64(dW), b["dW"]) <= GRAD_RFRO
    # and against the whole-vocabulary call on the same GPU
    with cta_pair(pair):
        loss1, lse1 = lce.forward(h, W, y)
        dH1, dW1 = lce.backward(h, W, y, lse1, dloss, chunk_rows=chunk)
    assert abs(loss.item() - loss1.item()) <= 1e-5 * abs(loss1.item())
    assert torch.max(torch.abs(lse - lse1)).item() <= 1e-4
    # lse differs in the last bits, which flips a few bf16 roundings of G;
    # kept exponentials are rounded to bf16 before the rescale
    assert rel_fro(to64(dW), to64(dW1)) <= (4e-3 if keep else 1e-3)
    # dH1 is rounded to bf16 once; the fp32 sum of partials is not
    assert rel_fro(to64(dH), to64(dH1)) <= 4e-3


def test_labels_out_of_range_and_in_other_slices():
    h, W, y = _inputs("bad", 260, 32, 600)
    y[3] = 600          # past the whole vocabulary: an error, row ignored
    y[9] = -5
    y[10] = 599         # last id, in the second slice only
    sizes = [300, 300]
    stats = []
    for k, (v0, Vs) in enumerate(_bounds(sizes)):
        stats.append(torch.stack(B.forward_slice(h, W[v0:v0 + Vs], y, v0,
                                                 600)))
        assert B.get_error() == B.LCE_ERR_LABEL_RANGE
    allst = torch.stack(stats)
    loss, lse = B.combine_slices(allst[:, 0].contiguous(),
                                 allst[:, 1].contiguous(),
                                 allst[:, 2].contiguous(), y, 600)
    assert B.get_error() == B.LCE_ERR_LABEL_RANGE
    f = oracle.forward(h.cpu(), W.cpu(), y.cpu())
    assert f["status"] == oracle.LABEL_RANGE
    assert abs(loss.item() - f["loss"]) <= LOSS_RTOL * abs(f["loss"])
    assert np.max(np.abs(to64(lse) - f["lse"])) <= LSE_ATOL
    assert allst[0, 2, 10].item() == 0.0 and allst[1, 2, 10].item() != 0.0


def test_module_without_group_is_one_slice():
    h, W, y = _inputs("one", 384, 64, 2000)
    d = torch.full((), 1.0, device=h.device)
    loss, lse = vp.forward(h, W, y, 0, 2000)
    dH, dW = vp.backward(h, W, y, lse, d, 0, 2000)
    loss1, lse1 = lce.forward(h, W, y)
    dH1, dW1 = lce.backward(h, W, y, lse1, d)
    assert lce.get_error() == 0
    assert abs(loss.item() - loss1.item()) <= 1e-6 * abs(loss1.item())
    assert torch.max(torch.abs(lse - lse1)).item() <= 1e-5
    assert rel_fro(to64(dW), to64(dW1)) <= 1e-3
    assert rel_fro(to64(dH), to64(dH1)) <= 4e-3


def test_module_keep_exp_matches_recompute():
    h, W, y = _inputs("mod", 384, 64, 2000)
    d = torch.full((), 0.75, device=h.device)
    ws = vp.exp_workspace(h, W[:1000])
    loss, lse = vp.forward_exp(h, W[:1000], y, 0, 2000, ws)
    dH, dW = vp.backward_exp(h, W[:1000], y, lse, d, 0, 2000, ws)
    # the single process holds only the first half of the vocabulary here,
    # so compare with the recomputing slice calls on the same half
    m, s, zy = B.forward_slice(h, W[:1000], y, 0, 2000)
    loss1, lse1 = B.combine_slices(m[None], s[None], zy[None], y, 2000)
    dH1, dW1 = B.backward_slice(h, W[:1000], y, lse1, d, 0, 2000)
    assert lce.get_error() == 0
    assert abs(loss.item() - loss1.item()) <= 1e-6 * abs(loss1.item())
    assert torch.max(torch.abs(lse - lse1)).item() <= 1e-5
    assert rel_fro(to64(dW), to64(dW1)) <= 4e-3
    assert rel_fro(to64(dH), to64(dH1)) <= 4e-3


@pytest.mark.parametrize("keep", [False, True], ids=["recompute", "keep_exp"])
def test_autograd_function_one_slice(keep):
    """With no group the one slice is the whole vocabulary: the autograd
    Function's loss and gradients equal the whole-vocabulary calls'."""
    h, W, y = _inputs("ag", 320, 64, 1500)
    hl = h.clone().requires_grad_(True)
    Wl = W.clone().requires_grad_(True)
    loss = vp.vocab_parallel_cross_entropy(hl, Wl, y, 0, 1500,
                                           keep_exp=keep)
    (2.0 * loss).backward()
    d = torch.full((), 2.0, device=h.device)
    loss1, lse1 = lce.forward(h, W, y)
    dH1, dW1 = lce.backward(h, W, y, lse1, d)
    assert lce.get_error() == 0
    assert abs(loss.item() - loss1.item()) <= 1e-6 * abs(loss1.item())
    assert hl.grad.dtype == h.dtype and Wl.grad.dtype == W.dtype
    assert rel_fro(to64(hl.grad), to64(dH1)) <= 8e-3
    assert rel_fro(to64(Wl.grad), to64(dW1)) <= 8e-3


# Loss variants (label smoothing eps, z-loss coefficient) in the
# vocabulary-parallel form: merged over the slices, the smoothed cross
# entropy plus the z-loss of the whole vocabulary, against the float64
# oracle's variant (the reading: target (1 - eps) onehot + eps / V_total,
# coef * lse^2 per valid row).
SLICE_VARIANTS = [(0.1, 0.0), (0.0, 1e-2), (0.2, 1e-3)]


@pytest.mark.parametrize("keep", [False, True], ids=["recompute", "keep_exp"])
@pytest.mark.parametrize("eps,zc", SLICE_VARIANTS,
                         ids=[f"eps{e}-z{z}" for e, z in SLICE_VARIANTS])
@pytest.mark.parametrize("name,L,H,V,sizes,chunk", CASES[:2],
                         ids=[c[0] for c in CASES[:2]])
def test_slices_with_loss_variant(name, L, H, V, sizes, chunk, eps, zc,
                                  keep):
    h, W, y = _inputs(name, L, H, V)
    hc, Wc, yc = h.cpu(), W.cpu(), y.cpu()
    dloss = torch.full((), 0.5, device=h.device)
    var = dict(label_smoothing=eps, z_loss=zc)
    wss = [B.slice_exp_workspace(L, H, Vs, h.dtype, h.device) if keep
           else None for _, Vs in _bounds(sizes)]
    stats = []
    for k, (v0, Vs) in enumerate(_bounds(sizes)):
        if keep:
            rows = B.forward_slice_exp(h, W[v0:v0 + Vs], y, v0, V, wss[k],
                                       **var)
        else:
            rows = B.forward_slice(h, W[v0:v0 + Vs], y, v0, V, **var)
        assert len(rows) == (4 if eps else 3)
        if eps:
            # the slice's logit sums against their definition in float64,
            # sum_j z_ij = sum_j h_i . W_j over the slice's columns
            z = hc.double() @ Wc[v0:v0 + Vs].double().T
            err = (rows[3].double().cpu() - z.sum(1)).abs()
            assert torch.all(err <= 1e-5 * z.abs().sum(1) + 1e-4)
        stats.append(torch.stack(rows))
    allst = torch.stack(stats)
    col = [allst[:, r].contiguous() for r in range(allst.shape[1])]
    loss, lse = B.combine_slices(col[0], col[1], col[2], y, V,
                                 zsum=col[3] if eps else None, **var)
    dH = torch.zeros(L, H, dtype=torch.float32, device=h.device)
    dWs = []
    for k, (v0, Vs) in enumerate(_bounds(sizes)):
        if keep:
            dH_part, dW_s = B.backward_slice_exp(h, W[v0:v0 + Vs], y, lse,
                                                 dloss, v0, V, wss[k], **var)
        else:
            dH_part, dW_s = B.backward_slice(h, W[v0:v0 + Vs], y, lse, dloss,
                                             v0, V, chunk_rows=chunk, **var)
        dH += dH_part
        dWs.append(dW_s)
    dW = torch.cat(dWs)
    assert lce.get_error() == 0
    fb = oracle.forward_backward(hc, Wc, yc, dloss=0.5, **var)
    assert abs(loss.item() - fb["loss"]) <= LOSS_RTOL * abs(fb["loss"])
    assert np.max(np.abs(to64(lse) - fb["lse"])) <= LSE_ATOL
    assert rel_fro(to64(dH), fb["dH"]) <= GRAD_RFRO
    assert rel_fro(to64(dW), fb["dW"]) <= GRAD_RFRO


def test_slice_ex_calls_with_zero_options_are_the_plain_calls():
    """The _ex slice calls given {0, 0} (and the logit sums anyway) give
    the plain calls' bits; the logit sums are written but do not enter."""
    import ctypes
    h, W, y = _inputs("zero_opts", 300, 64, 1000)
    lib = lce.load()
    zero = ctypes.pointer(B.LossOpts(0.0, 0.0))
    L, H = h.shape
    v0, Vs, V = 333, 333, 1000
    Ws = W[v0:v0 + Vs].contiguous()
    plain = B.forward_slice(h, Ws, y, v0, V)
    ws = B.alloc_workspace(L, H, Vs, h.dtype, 0, h.device)
    out = torch.empty(4, L, dtype=torch.float32, device=h.device)
    st = lib.lce_forward_slice_ex(
        h.data_ptr(), Ws.data_ptr(), B.LCE_BF16, y.data_ptr(), L, H, Vs, v0,
        V, -100, zero, out[0].data_ptr(), out[1].data_ptr(),
        out[2].data_ptr(), out[3].data_ptr(), ws.data_ptr(), ws.numel(),
        torch.cuda.current_stream().cuda_stream)
    assert st == 0
    for a, b in zip(plain, out[:3]):
        assert torch.equal(a, b)
    z = h.cpu().double() @ Ws.cpu().double().T
    err = (out[3].double().cpu() - z.sum(1)).abs()
    assert torch.all(err <= 1e-5 * z.abs().sum(1) + 1e-4)
    # combine: the plain call and the _ex call with zsum and {0, 0}
    loss0, lse0 = B.combine_slices(plain[0][None], plain[1][None],
                                   plain[2][None], y, V)
    cws = torch.empty(lib.lce_combine_workspace_size(L), dtype=torch.uint8,
                      device=h.device)
    loss1 = torch.empty((), dtype=torch.float32, device=h.device)
    lse1 = torch.empty(L, dtype=torch.float32, device=h.device)
    st = lib.lce_combine_slices_ex(
        out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(),
        out[3].data_ptr(), 1, y.data_ptr(), L, V, -100, zero,
        loss1.data_ptr(), lse1.data_ptr(), cws.data_ptr(), cws.numel(),
        torch.cuda.current_stream().cuda_stream)
    assert st == 0
    assert torch.equal(loss0, loss1) and torch.equal(lse0, lse1)
    assert lce.get_error() == 0


@pytest.mark.parametrize("keep", [False, True], ids=["recompute", "keep_exp"])
def test_autograd_function_one_slice_with_variant(keep):
    """With no group and a loss variant, the autograd Function's loss and
    gradients equal the whole-vocabulary variant calls'."""
    h, W, y = _inputs("ag_var", 320, 64, 1500)
    var = dict(label_smoothing=0.15, z_loss=2e-3)
    hl = h.clone().requires_grad_(True)
    Wl = W.clone().requires_grad_(True)
    loss = vp.vocab_parallel_cross_entropy(hl, Wl, y, 0, 1500,
                                           keep_exp=keep, **var)
    (2.0 * loss).backward()
    d = torch.full((), 2.0, device=h.device)
    loss1, lse1 = lce.forward(h, W, y, **var)
    dH1, dW1 = lce.backward(h, W, y, lse1, d, **var)
    assert lce.get_error() == 0
    assert abs(loss.item() - loss1.item()) <= 1e-6 * abs(loss1.item())
    assert rel_fro(to64(hl.grad), to64(dH1)) <= 8e-3
    assert rel_fro(to64(Wl.grad), to64(dW1)) <= 8e-3


@pytest.mark.parametrize("keep", [False, True], ids=["recompute", "keep_exp"])
def test_slice_optional_gradients(keep):
    """A frozen head slice (W_slice without grad) computes only dH, with
    the bits of the full call's dH; a frozen input only the slice's dW."""
    h, W, y = _inputs("opt_slice", 320, 64, 1500)
    d = torch.full((), 1.0, device=h.device)
    Ws = W[:1000].contiguous()
    if keep:
        ws = vp.exp_workspace(h, Ws)
        _, lse = vp.forward_exp(h, Ws, y, 0, 1500, ws)
        full = vp.backward_exp(h, Ws, y, lse, d, 0, 1500, ws)
        vp.forward_exp(h, Ws, y, 0, 1500, ws)
        only_dH = vp.backward_exp(h, Ws, y, lse, d, 0, 1500, ws,
                                  compute_dW=False)
        vp.forward_exp(h, Ws, y, 0, 1500, ws)
        only_dW = vp.backward_exp(h, Ws, y, lse, d, 0, 1500, ws,
                                  compute_dH=False)
    else:
        _, lse = vp.forward(h, Ws, y, 0, 1500)
        full = vp.backward(h, Ws, y, lse, d, 0, 1500)
        only_dH = vp.backward(h, Ws, y, lse, d, 0, 1500, compute_dW=False)
        only_dW = vp.backward(h, Ws, y, lse, d, 0, 1500, compute_dH=False)
    assert only_dH[1] is None and only_dW[0] is None
    assert torch.equal(only_dH[0], full[0])
    assert torch.equal(only_dW[1], full[1])
    hh = h.clone().requires_grad_(True)
    loss = vp.vocab_parallel_cross_entropy(hh, Ws, y, 0, 1500, keep_exp=keep)
    loss.backward()
    assert torch.equal(hh.grad, full[0].to(h.dtype))
    assert lce.get_error() == 0
