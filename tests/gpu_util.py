"""Helpers shared by the GPU tests: tolerances and comparisons.

Tolerances of the comparison with the float64 oracle, fixed for this
library (bf16 operands, fp32 accumulation):
  loss        relative error <= 1e-3
  dH, dW      relative Frobenius error <= 1e-2
  lse         max abs error <= 2e-3 (bf16 inputs: the oracle sees the same
              bf16 values; fp32 inputs: the GPU rounds them to bf16 first)
"""
import numpy as np
import pytest
import torch

LOSS_RTOL = 1e-3
GRAD_RFRO = 1e-2
LSE_ATOL = 2e-3


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import chunked_lm_head_gemm_gb300 as lce
    lce.load(build_if_missing=True)
    return torch.device("cuda:0")


def rel_fro(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(got - ref)
    return float(num / den) if den > 0 else float(num)


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


MODES = ["separate", "fused"]
# contraction variants under test: single CTAs (128 x 256 tiles) and CTA
# pairs (tcgen05 cta_group::2, 256 x 256 tiles; the library's default)
PAIRS = [False, True]


class cta_pair:
    """Context: run the library's contractions on CTA pairs or single CTAs
    (None leaves the process setting alone)."""

    def __init__(self, pair):
        self.pair = pair

    def __enter__(self):
        from chunked_lm_head_gemm_gb300 import _binding as B
        self.before = B.get_cta_pair()
        if self.pair is not None:
            B.set_cta_pair(self.pair)

    def __exit__(self, *exc):
        from chunked_lm_head_gemm_gb300 import _binding as B
        B.set_cta_pair(self.before)


def run_gpu(h, W, y, dloss=1.0, chunk_rows=0, ignore_index=-100,
            mode="separate", pair=None, **variant):
    """Forward + backward through the library; returns host float64 arrays.

    mode "separate": lce_forward then lce_backward (logits recomputed);
    mode "fused": lce_forward_backward, then lce_scale_gradients by dloss.
    pair: True/False selects CTA-pair or single-CTA contractions.
    variant: label_smoothing / z_loss (the _ex calls)."""
    with cta_pair(pair):
        return _run_gpu(h, W, y, dloss, chunk_rows, ignore_index, mode,
                        variant)


def _run_gpu(h, W, y, dloss, chunk_rows, ignore_index, mode, variant):
    import chunked_lm_head_gemm_gb300 as lce
    d = torch.full((), float(dloss), device=h.device)
    if mode == "fused":
        loss, lse, dH, dW = lce.forward_backward(h, W, y, ignore_index,
                                                 chunk_rows, **variant)
        lce.scale_gradients(dH, dW, d)
    else:
        loss, lse = lce.forward(h, W, y, ignore_index, **variant)
        dH, dW = lce.backward(h, W, y, lse, d, ignore_index, chunk_rows,
                              **variant)
    status = lce.get_error()
    return dict(loss=float(loss.item()), lse=to64(lse), dH=to64(dH),
                dW=to64(dW), status=status)


def assert_parity(gpu, f, b, lse_atol=LSE_ATOL, check_dW=True, dW_rows=None):
    assert abs(gpu["loss"] - f["loss"]) <= LOSS_RTOL * max(abs(f["loss"]), 1e-30), \
        f"loss {gpu['loss']} vs oracle {f['loss']}"
    err = np.max(np.abs(gpu["lse"] - f["lse"]))
    assert err <= lse_atol, f"lse max abs err {err}"
    e = rel_fro(gpu["dH"], b["dH"])
    assert e <= GRAD_RFRO, f"dH rel Frobenius err {e}"
    if check_dW:
        got = gpu["dW"] if dW_rows is None else gpu["dW"][dW_rows]
        e = rel_fro(got, b["dW"])
        assert e <= GRAD_RFRO, f"dW rel Frobenius err {e}"
