"""Pins of the float64 gated-MLP oracle (the sequence-tiled MLP workload).

The oracle computes y = (silu(x Wg^T) * (x Wu^T)) Wd^T and its backward
("Training Beyond 1M Tokens", section "One GPU is not enough: split the
sequence across many": one MLP line is
down_proj(act_fn(gate_proj(x)) * up_proj(x)); act_fn = SiLU, Qwen3's). It is
checked against things it shares no code with:

* PyTorch float64 autograd through torch.nn.functional.silu;
* central finite differences of <y, dy>;
* closed forms: Wu = 0 and Wg = 0 (silu(0) = 0, silu'(0) = 1/2);
* the row-tiling exactness the guide relies on: rows are independent in
  y and dx, and the weight gradients are sums of per-tile pieces.
"""
import numpy as np
import pytest
import torch


def _problem(L, H, I, seed, scale=0.5):
    rs = np.random.default_rng(seed)
    x = rs.standard_normal((L, H))
    Wg = rs.standard_normal((I, H)) * scale
    Wu = rs.standard_normal((I, H)) * scale
    Wd = rs.standard_normal((H, I)) * scale
    dy = rs.standard_normal((L, H))
    return x, Wg, Wu, Wd, dy


def _torch_ref(x, Wg, Wu, Wd, dy):
    t = [torch.tensor(a, requires_grad=True) for a in (x, Wg, Wu, Wd)]
    xt, gt, ut, dt = t
    y = (torch.nn.functional.silu(xt @ gt.T) * (xt @ ut.T)) @ dt.T
    y.backward(torch.tensor(dy))
    return y.detach().numpy(), [a.grad.numpy() for a in t]


@pytest.mark.parametrize("L,H,I,seed", [(1, 1, 1, 0), (5, 3, 7, 1),
                                        (33, 16, 40, 2)])
def test_against_torch_autograd(oracle_mod, L, H, I, seed):
    x, Wg, Wu, Wd, dy = _problem(L, H, I, seed)
    y, (dx, dWg, dWu, dWd) = _torch_ref(x, Wg, Wu, Wd, dy)
    r = oracle_mod.mlp(x, Wg, Wu, Wd, dy)
    np.testing.assert_allclose(r["y"], y, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["dx"], dx, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(r["dWg"], dWg, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(r["dWu"], dWu, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(r["dWd"], dWd, rtol=1e-11, atol=1e-13)


def test_bf16_inputs_widened_exactly(oracle_mod):
    x, Wg, Wu, Wd, dy = _problem(6, 8, 12, 3)
    tb = [torch.tensor(a).to(torch.bfloat16) for a in (x, Wg, Wu, Wd)]
    y, grads = _torch_ref(*[a.double().numpy() for a in tb], dy)
    r = oracle_mod.mlp(*tb, dy=dy)
    np.testing.assert_allclose(r["y"], y, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["dWd"], grads[3], rtol=1e-11, atol=1e-13)


def test_finite_differences(oracle_mod):
    x, Wg, Wu, Wd, dy = _problem(4, 3, 5, 4)
    r = oracle_mod.mlp(x, Wg, Wu, Wd, dy)
    eps = 1e-6
    rs = np.random.default_rng(9)

    def f(xx, gg, uu, dd):
        return float(np.sum(oracle_mod.mlp(xx, gg, uu, dd)["y"] * dy))

    arrays = [x, Wg, Wu, Wd]
    grads = [r["dx"], r["dWg"], r["dWu"], r["dWd"]]
    for which in range(4):
        for _ in range(5):
            a = arrays[which]
            idx = tuple(rs.integers(0, n) for n in a.shape)
            plus = [v.copy() for v in arrays]
            minus = [v.copy() for v in arrays]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            fd = (f(*plus) - f(*minus)) / (2 * eps)
            assert fd == pytest.approx(grads[which][idx], rel=1e-6, abs=1e-8)


def test_up_projection_zero(oracle_mod):
    """Wu = 0: u = 0, so y = 0, dWd = 0, dg = 0 and dx = 0; only
    du = (dy Wd) * silu(x Wg^T) survives, in dWu = du^T x."""
    x, Wg, Wu, Wd, dy = _problem(7, 5, 9, 5)
    Wu[:] = 0.0
    r = oracle_mod.mlp(x, Wg, Wu, Wd, dy)
    assert np.all(r["y"] == 0.0) and np.all(r["dWd"] == 0.0)
    assert np.all(r["dx"] == 0.0) and np.all(r["dWg"] == 0.0)
    g = x @ Wg.T
    du = (dy @ Wd) * (g / (1.0 + np.exp(-g)))
    np.testing.assert_allclose(r["dWu"], du.T @ x, rtol=1e-12, atol=1e-13)


def test_gate_projection_zero(oracle_mod):
    """Wg = 0: g = 0, silu(0) = 0 and silu'(0) = 1/2, so y = 0, du = 0 and
    dg = (dy Wd) * u / 2."""
    x, Wg, Wu, Wd, dy = _problem(6, 4, 8, 6)
    Wg[:] = 0.0
    r = oracle_mod.mlp(x, Wg, Wu, Wd, dy)
    assert np.all(r["y"] == 0.0) and np.all(r["dWu"] == 0.0)
    dg = (dy @ Wd) * (x @ Wu.T) * 0.5
    np.testing.assert_allclose(r["dWg"], dg.T @ x, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["dx"], dg @ Wg, rtol=1e-12, atol=1e-13)


def test_row_tiles_add_up(oracle_mod):
    """The guide's sequence tiling: per-tile y and dx are the whole's rows;
    per-tile weight gradients sum to the whole's."""
    x, Wg, Wu, Wd, dy = _problem(20, 6, 10, 7)
    whole = oracle_mod.mlp(x, Wg, Wu, Wd, dy)
    acc = {k: 0.0 for k in ("dWg", "dWu", "dWd")}
    for r0 in range(0, 20, 6):
        part = oracle_mod.mlp(x[r0:r0 + 6], Wg, Wu, Wd, dy[r0:r0 + 6])
        np.testing.assert_allclose(part["y"], whole["y"][r0:r0 + 6],
                                   rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(part["dx"], whole["dx"][r0:r0 + 6],
                                   rtol=1e-14, atol=1e-15)
        for k in acc:
            acc[k] = acc[k] + part[k]
    for k in acc:
        np.testing.assert_allclose(acc[k], whole[k], rtol=1e-12, atol=1e-13)
