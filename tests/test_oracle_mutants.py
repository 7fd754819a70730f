"""Planted mistakes in the oracle must be caught by its pins.

Each case copies lce_oracle.c, plants one plausible mistake (a dropped
term, a wrong sign, a wrong index, a transposed operand, a wrong
normaliser), compiles the copy into a temporary library and checks that
the pins of tests/test_oracle_pins.py reject it. Runs on the CPU only.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from tests import test_oracle_pins as pins

MLP_MUTANTS = {
    "silu_grad_sign": ("return s * (1.0 + t * (1.0 - s));",
                       "return s * (1.0 + t * s);"),
    "du_uses_grad": ("j->du[r * j->I + i] = da * silu(g);",
                     "j->du[r * j->I + i] = da * silu_grad(g);"),
    "dx_drops_up": ("dxr[k] += cg * wg[k] + cu * wu[k];",
                    "dxr[k] += cg * wg[k];"),
    "dWd_transposed": ("double c = j->dy[r * j->H + h];",
                       "double c = j->dy[r * j->H + (h + 1) % j->H];"),
    "gate_up_swapped": ("j->a[r * j->I + i] = silu(sg) * su;",
                        "j->a[r * j->I + i] = silu(su) * sg;"),
    "da_wrong_index": ("for (int64_t h = 0; h < j->H; ++h) da += dyr[h] * j->Wd[h * j->I + i];",
                       "for (int64_t h = 0; h < j->H; ++h) da += dyr[h] * j->Wd[i * j->H + h % j->H];"),
}

MUTANTS = {
    "drop_onehot": ("g[y] -= jb->gscale;", "(void)y;"),
    "onehot_sign": ("g[y] -= jb->gscale;", "g[y] += jb->gscale;"),
    "lse_drops_max": ("return m + log(s);", "return log(s);"),
    "softmax_unshifted": ("g[j] = jb->gscale * exp(z[j] - lse);",
                          "g[j] = jb->gscale * exp(z[j]);"),
    "dot_wrong_index": ("acc += x[k] * (double)f;",
                        "acc += x[(k + 1) % H] * (double)f;"),
    "dot_wrong_index_f64": ("for (int64_t k = 0; k < H; ++k) acc += x[k] * w[k];",
                            "for (int64_t k = 0; k < H; ++k) acc += x[k] * w[H - 1 - k];"),
    "dW_transposed": ("const double *hr = jb->hd + i * jb->H;",
                      "const double *hr = jb->hd + (j % jb->L) * jb->H;"),
    "dH_uses_h": ("if (g[j] != 0.0) axpy_row(g[j], jb->W, jb->dtype, j, jb->H, out);",
                  "if (g[j] != 0.0) axpy_row(g[j], jb->W, jb->dtype, (j + 1) % jb->V, jb->H, out);"),
    "mean_over_all_rows": ("if (loss) *loss = n > 0 ? total / (double)n : 0.0;",
                           "if (loss) *loss = n > 0 ? total / (double)L : 0.0;"),
    "grad_scale_all_rows": ("proto.gscale = n > 0 ? dloss / (double)n : 0.0;\n        st = run_rows(proto, L, nthreads);",
                            "proto.gscale = n > 0 ? dloss / (double)L : 0.0;\n        st = run_rows(proto, L, nthreads);"),
    "ignored_rows_count": ("if (label_is_valid(labels[i], V, ignore_index))\n            ++n;",
                           "if (labels[i] != ignore_index || 1)\n            ++n;"),
    # the loss variants (label smoothing, z-loss)
    "smooth_loss_over_V_minus_1": ("double q = (j == y ? 1.0 - eps : 0.0) + eps / (double)V;",
                                   "double q = (j == y ? 1.0 - eps : 0.0) + eps / (double)(V - 1);"),
    "smooth_grad_over_V_minus_1": ("const double qu = jb->eps / (double)jb->V;",
                                   "const double qu = jb->eps / (double)(jb->V - 1);"),
    "smooth_onehot_not_scaled": ("g[y] -= jb->gscale * (1.0 - jb->eps);",
                                 "g[y] -= jb->gscale;"),
    "z_loss_missing_in_loss": ("return t + zcoef * lse * lse;", "return t;"),
    "z_loss_grad_factor": ("const double zf = 1.0 + 2.0 * jb->zcoef * lse;",
                           "const double zf = 1.0 + jb->zcoef * lse;"),
}

PIN_CHECKS = [
    lambda o: pins.test_hand_worked_example(o),
    lambda o: pins.test_against_torch_cross_entropy_f64(o, 37, 19, 53, 2),
    lambda o: pins.test_low_precision_inputs_are_widened_exactly(
        o, pins.torch.bfloat16),
    lambda o: pins.test_finite_differences(o),
    lambda o: pins.test_w_zero_closed_form(o, 4096),
    lambda o: pins.test_v2_is_logistic_loss(o),
    lambda o: pins.test_invariants(o),
    lambda o: pins.test_all_ignored_and_bad_labels(o),
    lambda o: pins.test_variants_against_torch_f64(o, 37, 19, 53, 2, 0.2,
                                                   0.05),
    lambda o: pins.test_variant_finite_differences(o),
    lambda o: pins.test_variant_w_zero_closed_form(o, 0.3, 1e-3),
]


def _caught(mod) -> bool:
    for check in PIN_CHECKS:
        try:
            check(mod)
        except (AssertionError, RuntimeError):
            return True
    return False


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new, 1))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread",
                    "-o", str(so), str(mutant), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_lib", oracle.load_library(str(so)))
    assert _caught(oracle), f"planted mistake {name} passed every pin"


def test_unmutated_passes_all_pins(oracle_mod):
    assert not _caught(oracle_mod)


def _mlp_caught(mod) -> bool:
    from tests import test_mlp_oracle_pins as mp
    checks = [
        lambda o: mp.test_against_torch_autograd(o, 5, 3, 7, 1),
        lambda o: mp.test_finite_differences(o),
        lambda o: mp.test_up_projection_zero(o),
        lambda o: mp.test_gate_projection_zero(o),
    ]
    for check in checks:
        try:
            check(mod)
        except (AssertionError, RuntimeError):
            return True
    return False


@pytest.mark.parametrize("name", sorted(MLP_MUTANTS))
def test_planted_mlp_mistake_is_caught(name, tmp_path, monkeypatch):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src_path = os.path.join(os.path.dirname(oracle._SRC), "mlp_oracle.c")
    src = open(src_path).read()
    old, new = MLP_MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutant = tmp_path / "mlp_mutant.c"
    mutant.write_text(src.replace(old, new, 1))
    so = tmp_path / "libmlpmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread",
                    "-o", str(so), oracle._SRC, str(mutant), "-lm"],
                   check=True)
    monkeypatch.setattr(oracle, "_lib", oracle.load_library(str(so)))
    assert _mlp_caught(oracle), f"planted mistake {name} passed every pin"


def test_unmutated_mlp_passes_all_pins(oracle_mod):
    assert not _mlp_caught(oracle_mod)
