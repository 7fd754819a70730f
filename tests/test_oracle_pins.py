"""Pins of the float64 oracle against things other than itself.

The oracle computes the plain definition of the chunked LM-head loss
("Training Beyond 1M Tokens", sections "The loss is the first thing to
break" and "The massive logits matrix: chunk it"). Each test below checks it
against something it does not share code with:

* a worked example solved by hand (tests/golden/hand_example.json);
* PyTorch's float64 cross_entropy with autograd (a library routine: the
  plain unchunked loss the pages name as the alternative);
* central finite differences of the oracle's own loss (gradients);
* the W = 0 closed form (tests/golden/w_zero.json);
* V = 2, where the loss is the logistic loss log1p(exp(z_other - z_y));
* invariants of the mathematics: gradient rows sum to zero, a common shift
  of all logits changes nothing but lse, row permutation, linearity in
  dloss, all-ignored rows.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rand_problem(L, H, V, seed, ignore_frac=0.2, dtype=np.float64,
                  w_std=0.5):
    rs = np.random.default_rng(seed)
    h = rs.standard_normal((L, H)).astype(dtype)
    W = (rs.standard_normal((V, H)) * w_std).astype(dtype)
    y = rs.integers(0, V, L).astype(np.int64)
    n_ign = int(round(ignore_frac * L))
    y[rs.permutation(L)[:n_ign]] = -100
    return h, W, y


def _torch_ref(h, W, y, dloss=1.0):
    ht = torch.tensor(np.asarray(h, dtype=np.float64), requires_grad=True)
    Wt = torch.tensor(np.asarray(W, dtype=np.float64), requires_grad=True)
    yt = torch.tensor(y)
    z = ht @ Wt.T
    loss = torch.nn.functional.cross_entropy(z, yt, ignore_index=-100,
                                             reduction="mean")
    (loss * dloss).backward()
    lse = torch.logsumexp(z.detach(), dim=1)
    return loss.item(), lse.numpy(), ht.grad.numpy(), Wt.grad.numpy()


def test_hand_worked_example(oracle_mod):
    g = json.load(open(os.path.join(GOLD, "hand_example.json")))
    h = np.array(g["h"])
    W = np.array(g["W"])
    y = np.array(g["labels"], dtype=np.int64)
    ex = g["expected"]
    f = oracle_mod.forward(h, W, y)
    b = oracle_mod.backward(h, W, y, dloss=g["dloss"])
    assert f["n_valid"] == ex["n_valid"]
    np.testing.assert_allclose(f["lse"], ex["lse"], rtol=1e-15)
    assert f["loss"] == pytest.approx(ex["loss"], rel=1e-15)
    np.testing.assert_allclose(b["dH"], ex["dH"], rtol=1e-15, atol=1e-17)
    np.testing.assert_allclose(b["dW"], ex["dW"], rtol=1e-15, atol=1e-17)


@pytest.mark.parametrize("L,H,V,seed", [(1, 1, 1, 0), (3, 2, 5, 1),
                                        (37, 19, 53, 2), (64, 33, 257, 3)])
def test_against_torch_cross_entropy_f64(oracle_mod, L, H, V, seed):
    h, W, y = _rand_problem(L, H, V, seed, ignore_frac=0.2 if L > 1 else 0.0)
    if (y != -100).sum() == 0:
        y[0] = 0
    dloss = 0.7
    loss, lse, dH, dW = _torch_ref(h, W, y, dloss)
    f = oracle_mod.forward(h, W, y)
    b = oracle_mod.backward(h, W, y, dloss=dloss)
    assert f["loss"] == pytest.approx(loss, rel=1e-12, abs=1e-14)
    np.testing.assert_allclose(f["lse"], lse, rtol=1e-12)
    np.testing.assert_allclose(b["dH"], dH, rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(b["dW"], dW, rtol=1e-10, atol=1e-14)
    # the logit at the label, for rows that take part
    z = h @ W.T
    valid = y != -100
    np.testing.assert_allclose(f["zy"][valid], z[valid, y[valid]], rtol=1e-12,
                               atol=1e-14)
    assert np.all(np.isnan(f["zy"][~valid]))


@pytest.mark.parametrize("tdtype", [torch.bfloat16, torch.float32])
def test_low_precision_inputs_are_widened_exactly(oracle_mod, tdtype):
    """bf16 / fp32 inputs give the float64 answer on their exact values."""
    h, W, y = _rand_problem(16, 24, 40, 7)
    ht = torch.tensor(h).to(tdtype)
    Wt = torch.tensor(W).to(tdtype)
    loss, lse, dH, dW = _torch_ref(ht.double().numpy(), Wt.double().numpy(), y)
    f = oracle_mod.forward(ht, Wt, y)
    b = oracle_mod.backward(ht, Wt, y)
    assert f["loss"] == pytest.approx(loss, rel=1e-12)
    np.testing.assert_allclose(f["lse"], lse, rtol=1e-12)
    np.testing.assert_allclose(b["dH"], dH, rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(b["dW"], dW, rtol=1e-10, atol=1e-14)


def test_finite_differences(oracle_mod):
    L, H, V = 8, 4, 16
    h, W, y = _rand_problem(L, H, V, 11)
    b = oracle_mod.backward(h, W, y, dloss=1.0)
    eps = 1e-6
    rs = np.random.default_rng(5)

    def loss_of(hh, WW):
        return oracle_mod.forward(hh, WW, y)["loss"]

    for _ in range(12):
        i, k = rs.integers(0, L), rs.integers(0, H)
        hp, hm = h.copy(), h.copy()
        hp[i, k] += eps
        hm[i, k] -= eps
        fd = (loss_of(hp, W) - loss_of(hm, W)) / (2 * eps)
        assert fd == pytest.approx(b["dH"][i, k], rel=1e-6, abs=1e-9)
        j, k = rs.integers(0, V), rs.integers(0, H)
        Wp, Wm = W.copy(), W.copy()
        Wp[j, k] += eps
        Wm[j, k] -= eps
        fd = (loss_of(h, Wp) - loss_of(h, Wm)) / (2 * eps)
        assert fd == pytest.approx(b["dW"][j, k], rel=1e-6, abs=1e-9)


@pytest.mark.parametrize("V", [4096, 151936])
def test_w_zero_closed_form(oracle_mod, V):
    g = json.load(open(os.path.join(GOLD, "w_zero.json")))
    lnV = g["ln_V"][str(V)]
    assert lnV == math.log(V)
    L, H = 6, 8
    rs = np.random.default_rng(3)
    h = rs.standard_normal((L, H))
    W = np.zeros((V, H))
    y = rs.integers(0, V, L).astype(np.int64)
    y[2] = -100
    dloss = 1.3
    f = oracle_mod.forward(h, W, y)
    np.testing.assert_allclose(f["lse"], lnV, rtol=1e-15)
    assert f["loss"] == pytest.approx(lnV, rel=1e-15)
    b = oracle_mod.backward(h, W, y, dloss=dloss)
    assert np.all(b["dH"] == 0.0)
    valid = y != -100
    n = valid.sum()
    expect = np.tile((dloss / n) * h[valid].sum(0) / V, (V, 1))
    for i in np.nonzero(valid)[0]:
        expect[y[i]] -= (dloss / n) * h[i]
    np.testing.assert_allclose(b["dW"], expect, rtol=1e-12, atol=1e-15)


def test_v2_is_logistic_loss(oracle_mod):
    L, H = 50, 7
    h, W, y = _rand_problem(L, H, 2, 13, ignore_frac=0.0, w_std=1.0)
    z = h @ W.T
    d = z[np.arange(L), 1 - y] - z[np.arange(L), y]
    expect = np.mean(np.log1p(np.exp(d)))
    assert oracle_mod.forward(h, W, y)["loss"] == pytest.approx(expect,
                                                                rel=1e-13)
    # d loss / d z_other = sigmoid(d) / L; d loss / d z_y = -sigmoid(d) / L
    sig = 1.0 / (1.0 + np.exp(-d))
    Gz = np.zeros((L, 2))
    Gz[np.arange(L), 1 - y] = sig / L
    Gz[np.arange(L), y] = -sig / L
    b = oracle_mod.backward(h, W, y)
    np.testing.assert_allclose(b["dH"], Gz @ W, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(b["dW"], Gz.T @ h, rtol=1e-12, atol=1e-15)


def test_v1_gives_zero(oracle_mod):
    h, W, y = _rand_problem(5, 3, 1, 17, ignore_frac=0.0)
    f = oracle_mod.forward(h, W, y)
    np.testing.assert_allclose(f["lse"], (h @ W.T)[:, 0], rtol=1e-15)
    assert f["loss"] == 0.0
    b = oracle_mod.backward(h, W, y)
    assert np.all(b["dH"] == 0.0) and np.all(b["dW"] == 0.0)


def test_invariants(oracle_mod):
    L, H, V = 40, 12, 70
    h, W, y = _rand_problem(L, H, V, 21)
    f = oracle_mod.forward(h, W, y)
    b = oracle_mod.backward(h, W, y, dloss=1.0)
    # each row of G sums to zero, hence the columns of dW sum to zero
    np.testing.assert_allclose(b["dW"].sum(0), 0.0, atol=1e-14)
    # a common shift of one row's logits: W -> W + 1 u^T adds h.u to every
    # logit of the row; loss and dH are unchanged, lse moves by h.u, and dW
    # is unchanged because G's rows sum to zero
    u = np.random.default_rng(2).standard_normal(H)
    W2 = W + u[None, :]
    f2 = oracle_mod.forward(h, W2, y)
    b2 = oracle_mod.backward(h, W2, y)
    assert f2["loss"] == pytest.approx(f["loss"], rel=1e-12)
    np.testing.assert_allclose(f2["lse"], f["lse"] + h @ u, rtol=1e-12)
    np.testing.assert_allclose(b2["dH"], b["dH"], rtol=1e-9, atol=1e-14)
    np.testing.assert_allclose(b2["dW"], b["dW"], rtol=1e-9, atol=1e-14)
    # row permutation leaves the loss unchanged and permutes dH
    p = np.random.default_rng(4).permutation(L)
    f3 = oracle_mod.forward(h[p], W, y[p])
    b3 = oracle_mod.backward(h[p], W, y[p])
    assert f3["loss"] == pytest.approx(f["loss"], rel=1e-13)
    np.testing.assert_allclose(b3["dH"], b["dH"][p], rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(b3["dW"], b["dW"], rtol=1e-12, atol=1e-15)
    # gradients are linear in dloss; dloss = 0 gives exact zeros
    b4 = oracle_mod.backward(h, W, y, dloss=-2.5)
    np.testing.assert_allclose(b4["dH"], -2.5 * b["dH"], rtol=1e-13)
    b0 = oracle_mod.backward(h, W, y, dloss=0.0)
    assert np.all(b0["dH"] == 0.0) and np.all(b0["dW"] == 0.0)


def test_chunked_sum_equals_whole(oracle_mod):
    """The pages' exactness argument: per-chunk sums of row losses add up to
    the whole loss (the reduction divides by one global N)."""
    L, H, V = 60, 10, 33
    h, W, y = _rand_problem(L, H, V, 23)
    f = oracle_mod.forward(h, W, y)
    total = 0.0
    for c0 in range(0, L, 16):
        fc = oracle_mod.forward(h[c0:c0 + 16], W, y[c0:c0 + 16])
        total += fc["loss"] * fc["n_valid"]
    assert total / f["n_valid"] == pytest.approx(f["loss"], rel=1e-13)


def test_all_ignored_and_bad_labels(oracle_mod):
    h, W, y = _rand_problem(6, 4, 9, 29, ignore_frac=0.0)
    y_all = np.full(6, -100, dtype=np.int64)
    f = oracle_mod.forward(h, W, y_all)
    assert f["n_valid"] == 0 and f["loss"] == 0.0
    np.testing.assert_allclose(f["lse"], _torch_ref(h, W, y)[1], rtol=1e-13)
    b = oracle_mod.backward(h, W, y_all)
    assert np.all(b["dH"] == 0.0) and np.all(b["dW"] == 0.0)
    # an out-of-range label is reported and its row is ignored
    y_bad = y.copy()
    y_bad[1] = 9
    y_bad[3] = -7
    f = oracle_mod.forward(h, W, y_bad)
    assert f["status"] == oracle_mod.LABEL_RANGE
    y_ign = y.copy()
    y_ign[[1, 3]] = -100
    f_ign = oracle_mod.forward(h, W, y_ign)
    assert f["n_valid"] == 4 and f["loss"] == pytest.approx(f_ign["loss"],
                                                             rel=1e-15)
    assert oracle_mod.count_valid(y_bad, 9) == (4, True)
    assert oracle_mod.count_valid(y_ign, 9) == (4, False)


def test_rows_matches_whole(oracle_mod):
    L, H, V = 30, 9, 41
    h, W, y = _rand_problem(L, H, V, 31)
    f = oracle_mod.forward(h, W, y)
    b = oracle_mod.backward(h, W, y, dloss=0.9)
    r = np.array([0, 7, 29, 7, 13])
    s = oracle_mod.rows(h, W, y, r, dloss=0.9)
    np.testing.assert_allclose(s["lse"], f["lse"][r], rtol=1e-15)
    np.testing.assert_allclose(s["dH"], b["dH"][r], rtol=1e-13, atol=1e-16)
    np.testing.assert_array_equal(np.isnan(s["zy"]), np.isnan(f["zy"][r]))


def test_threads_do_not_change_results(oracle_mod):
    h, W, y = _rand_problem(23, 7, 19, 37)
    a = oracle_mod.backward(h, W, y, nthreads=1)
    b = oracle_mod.backward(h, W, y, nthreads=5)
    assert np.array_equal(a["dH"], b["dH"]) and np.array_equal(a["dW"],
                                                              b["dW"])


def test_dW_vocab_subset_matches_whole(oracle_mod):
    L, H, V = 20, 6, 31
    h, W, y = _rand_problem(L, H, V, 41)
    full = oracle_mod.backward(h, W, y, dloss=1.1)["dW"]
    v = np.array([30, 0, 5, 5, 17])
    sub = oracle_mod.backward(h, W, y, dloss=1.1, want_dH=False,
                              vrows=v)["dW"]
    np.testing.assert_array_equal(sub, full[v])


# ---- single pass and loss variants ------------------------------------------

VARIANTS = [(0.1, 0.0), (0.3, 0.0), (1.0, 0.0), (0.0, 1e-2), (0.2, 0.05)]


def _torch_variant_ref(h, W, y, eps, zcoef, dloss=1.0):
    """PyTorch float64: F.cross_entropy with label_smoothing (a library
    routine) plus zcoef * lse^2 averaged over the rows that take part, and
    autograd for the gradients."""
    ht = torch.tensor(np.asarray(h, dtype=np.float64), requires_grad=True)
    Wt = torch.tensor(np.asarray(W, dtype=np.float64), requires_grad=True)
    yt = torch.tensor(y)
    z = ht @ Wt.T
    loss = torch.nn.functional.cross_entropy(z, yt, ignore_index=-100,
                                             reduction="mean",
                                             label_smoothing=eps)
    valid = yt != -100
    lse = torch.logsumexp(z, dim=1)
    if zcoef:
        loss = loss + zcoef * (lse[valid] ** 2).sum() / valid.sum()
    (loss * dloss).backward()
    return loss.item(), lse.detach().numpy(), ht.grad.numpy(), Wt.grad.numpy()


@pytest.mark.parametrize("eps,zcoef", VARIANTS)
@pytest.mark.parametrize("L,H,V,seed", [(3, 2, 5, 1), (37, 19, 53, 2)])
def test_variants_against_torch_f64(oracle_mod, L, H, V, seed, eps, zcoef):
    h, W, y = _rand_problem(L, H, V, seed)
    if (y != -100).sum() == 0:
        y[0] = 0
    dloss = 0.7
    loss, lse, dH, dW = _torch_variant_ref(h, W, y, eps, zcoef, dloss)
    kw = dict(label_smoothing=eps, z_loss=zcoef)
    f = oracle_mod.forward(h, W, y, **kw)
    b = oracle_mod.backward(h, W, y, dloss=dloss, **kw)
    assert f["loss"] == pytest.approx(loss, rel=1e-12, abs=1e-14)
    np.testing.assert_allclose(f["lse"], lse, rtol=1e-12)
    np.testing.assert_allclose(b["dH"], dH, rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(b["dW"], dW, rtol=1e-10, atol=1e-14)
    r = np.array([0, L - 1])
    s = oracle_mod.rows(h, W, y, r, dloss=dloss, **kw)
    np.testing.assert_allclose(s["dH"], dH[r], rtol=1e-10, atol=1e-14)


def test_variant_finite_differences(oracle_mod):
    L, H, V = 8, 4, 16
    h, W, y = _rand_problem(L, H, V, 19)
    kw = dict(label_smoothing=0.2, z_loss=0.03)
    b = oracle_mod.backward(h, W, y, dloss=1.0, **kw)
    eps = 1e-6
    rs = np.random.default_rng(6)

    def loss_of(hh, WW):
        return oracle_mod.forward(hh, WW, y, **kw)["loss"]

    for _ in range(12):
        i, k = rs.integers(0, L), rs.integers(0, H)
        hp, hm = h.copy(), h.copy()
        hp[i, k] += eps
        hm[i, k] -= eps
        fd = (loss_of(hp, W) - loss_of(hm, W)) / (2 * eps)
        assert fd == pytest.approx(b["dH"][i, k], rel=1e-6, abs=1e-9)
        j, k = rs.integers(0, V), rs.integers(0, H)
        Wp, Wm = W.copy(), W.copy()
        Wp[j, k] += eps
        Wm[j, k] -= eps
        fd = (loss_of(h, Wp) - loss_of(h, Wm)) / (2 * eps)
        assert fd == pytest.approx(b["dW"][j, k], rel=1e-6, abs=1e-9)


@pytest.mark.parametrize("eps,zcoef", [(0.1, 0.0), (1.0, 0.0), (0.3, 1e-3)])
def test_variant_w_zero_closed_form(oracle_mod, eps, zcoef):
    """W = 0: every logit is 0, lse = ln V and the smoothed cross entropy of
    every row is ln V whatever eps (the target sums to one), so loss =
    ln V + zcoef (ln V)^2; dH = 0; dW[v] = dloss/N sum_valid ((1 + 2 zcoef
    ln V)/V - q_v) h_i with q_v = (1 - eps)[v == y_i] + eps/V."""
    V = 4096
    g = json.load(open(os.path.join(GOLD, "w_zero.json")))
    lnV = g["ln_V"][str(V)]
    L, H = 6, 8
    rs = np.random.default_rng(8)
    h = rs.standard_normal((L, H))
    W = np.zeros((V, H))
    y = rs.integers(0, V, L).astype(np.int64)
    y[4] = -100
    dloss = 0.9
    kw = dict(label_smoothing=eps, z_loss=zcoef)
    f = oracle_mod.forward(h, W, y, **kw)
    assert f["loss"] == pytest.approx(lnV + zcoef * lnV ** 2, rel=1e-13)
    b = oracle_mod.backward(h, W, y, dloss=dloss, **kw)
    assert np.all(b["dH"] == 0.0)
    valid = y != -100
    n = valid.sum()
    p = (1.0 + 2.0 * zcoef * lnV) / V
    expect = np.tile((dloss / n) * (p - eps / V) * h[valid].sum(0), (V, 1))
    for i in np.nonzero(valid)[0]:
        expect[y[i]] -= (dloss / n) * (1.0 - eps) * h[i]
    np.testing.assert_allclose(b["dW"], expect, rtol=1e-11, atol=1e-15)


def test_full_smoothing_does_not_depend_on_labels(oracle_mod):
    """eps = 1: the target is uniform, so which valid label a row has does
    not matter (only whether it is ignored)."""
    L, H, V = 30, 6, 25
    h, W, y = _rand_problem(L, H, V, 43)
    y2 = y.copy()
    valid = y != -100
    y2[valid] = (y[valid] + 7) % V
    kw = dict(label_smoothing=1.0)
    f = oracle_mod.forward(h, W, y, **kw)
    f2 = oracle_mod.forward(h, W, y2, **kw)
    assert f2["loss"] == pytest.approx(f["loss"], rel=1e-13)
    b = oracle_mod.backward(h, W, y, **kw)
    b2 = oracle_mod.backward(h, W, y2, **kw)
    np.testing.assert_allclose(b2["dW"], b["dW"], rtol=1e-12, atol=1e-16)


def test_smoothing_is_shift_invariant_and_z_loss_is_not(oracle_mod):
    """The smoothed target sums to one, so W -> W + 1 u^T changes neither
    the smoothed loss nor its gradients; the z-loss term moves with lse,
    which moves by h.u exactly."""
    L, H, V = 40, 12, 70
    h, W, y = _rand_problem(L, H, V, 47)
    u = np.random.default_rng(9).standard_normal(H)
    W2 = W + u[None, :]
    kw = dict(label_smoothing=0.3)
    f, f2 = (oracle_mod.forward(h, w, y, **kw) for w in (W, W2))
    assert f2["loss"] == pytest.approx(f["loss"], rel=1e-12)
    b, b2 = (oracle_mod.backward(h, w, y, **kw) for w in (W, W2))
    np.testing.assert_allclose(b2["dH"], b["dH"], rtol=1e-9, atol=1e-14)
    np.testing.assert_allclose(b2["dW"], b["dW"], rtol=1e-9, atol=1e-14)
    zc = 0.02
    g, g2 = (oracle_mod.forward(h, w, y, label_smoothing=0.3, z_loss=zc)
             for w in (W, W2))
    valid = y != -100
    s = (h @ u)[valid]
    lse = f["lse"][valid]
    moved = zc * np.mean((lse + s) ** 2 - lse ** 2)
    assert g2["loss"] - g["loss"] == pytest.approx(moved, rel=1e-9)


@pytest.mark.parametrize("eps,zcoef", [(0.0, 0.0), (0.2, 0.05)])
def test_single_pass_matches_forward_and_backward(oracle_mod, eps, zcoef):
    L, H, V = 33, 10, 47
    h, W, y = _rand_problem(L, H, V, 53)
    kw = dict(label_smoothing=eps, z_loss=zcoef)
    f = oracle_mod.forward(h, W, y, **kw)
    b = oracle_mod.backward(h, W, y, dloss=1.3, **kw)
    v = np.array([46, 0, 3])
    fb = oracle_mod.forward_backward(h, W, y, dloss=1.3, **kw)
    fbv = oracle_mod.forward_backward(h, W, y, dloss=1.3, vrows=v,
                                      want_dH=False, **kw)
    assert fb["loss"] == f["loss"] and fb["n_valid"] == f["n_valid"]
    assert np.array_equal(fb["lse"], f["lse"])
    assert np.array_equal(fb["dH"], b["dH"]) and np.array_equal(fb["dW"],
                                                               b["dW"])
    assert fbv["dH"] is None and np.array_equal(fbv["dW"], b["dW"][v])


def test_variant_arguments_are_checked(oracle_mod):
    h, W, y = _rand_problem(4, 3, 5, 59)
    for kw in (dict(label_smoothing=-0.1), dict(label_smoothing=1.5),
               dict(z_loss=-1.0), dict(z_loss=float("inf"))):
        with pytest.raises(RuntimeError):
            oracle_mod.forward(h, W, y, **kw)
