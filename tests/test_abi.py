"""The C ABI without a GPU: the library loads, exports every function that
include/lce.h declares, sizes its workspace, and rejects bad arguments
before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import chunked_lm_head_gemm_gb300 as lce
    return lce.load(build_if_missing=True)


def _declared():
    text = open(os.path.join(ROOT, "include", "lce.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lce_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = _declared()
    assert "lce_forward" in names and "lce_backward" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in lce.h but not exported"
    from chunked_lm_head_gemm_gb300 import _binding as B
    assert sorted(B.EXPORTED) == names


def test_status_strings(lib):
    for code, name in enumerate(["LCE_OK", "LCE_ERR_INVALID_ARG",
                                 "LCE_ERR_UNSUPPORTED", "LCE_ERR_WORKSPACE",
                                 "LCE_ERR_LABEL_RANGE", "LCE_ERR_TIMEOUT",
                                 "LCE_ERR_CUDA"]):
        assert lib.lce_status_string(code).decode() == name
    assert lib.lce_status_string(99).decode() == "LCE_ERR_UNKNOWN"


def test_workspace_size(lib):
    f = lib.lce_workspace_size
    assert f(0, 256, 4096, 0, 0) == 0          # L < 1
    assert f(512, 12, 4096, 0, 0) == 0         # H % 8 != 0
    assert f(512, 256, 4096, 7, 0) == 0        # bad dtype
    assert f(512, 256, 4096, 0, -1) == 0       # bad chunk
    small = f(512, 256, 4096, 0, 128)
    big = f(512, 256, 4096, 0, 512)
    assert 0 < small < big
    # fp32 inputs add bf16 copies of h and W
    assert f(512, 256, 4096, 1, 512) - big >= 2 * (512 * 256 + 4096 * 256)
    # the gradient-logit chunk dominates: chunk * round_up(V, 8) * 2 bytes
    L, H, V = 131072, 4096, 151936
    c = lib.lce_default_chunk_rows(L, H, V)
    assert c % 128 == 0 and 0 < c <= L
    assert f(L, H, V, 0, 0) >= c * V * 2
    # plus the forward statistics (16 splits x (max, sum, logit sum) + the
    # label logit) and the fused path's per-tile row maxima (chunk x
    # ceil(V/256) floats)
    tiles = -(-V // 256)
    assert f(L, H, V, 0, 0) < (c * V * 2 + (16 * 12 + 4 + 1) * L +
                               4 * c * tiles + (1 << 20))
    # peak extra memory is O(chunk * V), far below the L x V fp32 logits
    assert f(L, H, V, 0, 0) < L * V * 4 / 8


def test_bad_arguments_return_before_any_device_call(lib):
    """Every call here fails validation first, so no pointer is used."""
    p = ctypes.c_void_p(0x1000)  # aligned but never dereferenced
    null = ctypes.c_void_p(0)
    i = ctypes.c_int64
    # null h
    assert lib.lce_forward(null, p, 0, p, 8, 8, 8, -100, p, p, p, 1 << 30,
                           null) == 1
    # H not a multiple of 8
    assert lib.lce_forward(p, p, 0, p, 8, 12, 8, -100, p, p, p, 1 << 30,
                           null) == 1
    # unsupported dtype
    assert lib.lce_forward(p, p, 5, p, 8, 8, 8, -100, p, p, p, 1 << 30,
                           null) == 2
    # misaligned W
    assert lib.lce_forward(p, ctypes.c_void_p(0x1002), 0, p, 8, 8, 8, -100,
                           p, p, p, 1 << 30, null) == 1
    # workspace too small
    assert lib.lce_forward(p, p, 0, p, 8, 8, 8, -100, p, p, p, 16,
                           null) == 3
    assert lib.lce_backward(p, p, 0, p, p, 8, 8, 8, -100, p, 0, p, p, p, 16,
                            null) == 3
    # negative chunk
    assert lib.lce_backward(p, p, 0, p, p, 8, 8, 8, -100, p, -5, p, p, p,
                            1 << 30, null) == 1
    # label count: null output, misaligned labels, negative L, V < 1
    assert lib.lce_count_valid(p, 8, 8, -100, null, null) == 1
    assert lib.lce_count_valid(ctypes.c_void_p(0x1004), 8, 8, -100, p,
                               null) == 1
    assert lib.lce_count_valid(p, -1, 8, -100, p, null) == 1
    assert lib.lce_count_valid(p, 8, 0, -100, p, null) == 1
    # vocabulary slices: slice past the vocabulary, negative offset
    assert lib.lce_forward_slice(p, p, 0, p, 8, 8, 8, 4, 10, -100, p, p, p,
                                 p, 1 << 30, null) == 1
    assert lib.lce_forward_slice(p, p, 0, p, 8, 8, 8, -1, 10, -100, p, p, p,
                                 p, 1 << 30, null) == 1
    assert lib.lce_backward_slice(p, p, 0, p, p, 8, 8, 8, 4, 10, -100, p, 0,
                                  p, p, p, 1 << 30, null) == 1
    assert lib.lce_combine_slices(p, p, p, 0, p, 8, 10, -100, p, p, p,
                                  1 << 20, null) == 1
    assert lib.lce_combine_slices(p, p, p, 2, p, 8, 10, -100, p, p, p, 8,
                                  null) == 3
    assert lib.lce_forward_slice_exp(p, p, 0, p, 8, 8, 8, 4, 10, -100, p, p,
                                     p, p, 1 << 30, null) == 1
    assert lib.lce_backward_slice_exp(p, p, 0, p, p, 8, 8, 8, 0, 10, -100, p,
                                      p, p, p, 16, null) == 3
    assert lib.lce_slice_exp_workspace_size(0, 8, 8, 0) == 0
    # the kept exponentials dominate: L x round_up(Vs, 8) x 2 bytes
    assert lib.lce_slice_exp_workspace_size(1024, 64, 1000, 0) >= 1024 * 1000 * 2
    assert lib.lce_combine_workspace_size(0) == 0
    assert lib.lce_combine_workspace_size(300) == 256 + 2 * 8
    # loss variants: out-of-range options are refused before anything else
    from chunked_lm_head_gemm_gb300 import _binding as B
    for eps, zc in ((-0.1, 0.0), (1.5, 0.0), (0.0, -1.0),
                    (0.0, float("inf")), (float("nan"), 0.0)):
        o = ctypes.pointer(B.LossOpts(eps, zc))
        assert lib.lce_forward_ex(p, p, 0, p, 8, 8, 8, -100, o, p, p, p,
                                  1 << 30, null) == 1
        assert lib.lce_backward_ex(p, p, 0, p, p, 8, 8, 8, -100, o, p, 0, p,
                                   p, p, 1 << 30, null) == 1
        assert lib.lce_forward_backward_ex(p, p, 0, p, 8, 8, 8, -100, o, 0,
                                           p, p, p, p, p, 1 << 30, null) == 1
    ok = ctypes.pointer(B.LossOpts(0.1, 1e-4))
    assert lib.lce_forward_ex(p, p, 0, p, 8, 8, 8, -100, ok, p, p, p, 16,
                              null) == 3
    assert lib.lce_forward_ex(p, p, 0, p, 8, 8, 8, -100, None, p, p, p, 16,
                              null) == 3
    # loss variants on vocabulary slices: bad options are refused, and the
    # logit sums are required (and 4-byte aligned) under label smoothing
    smooth = ctypes.pointer(B.LossOpts(0.1, 0.0))
    zonly = ctypes.pointer(B.LossOpts(0.0, 1e-4))
    odd = ctypes.c_void_p(0x1002)
    for o in (ctypes.pointer(B.LossOpts(-0.1, 0.0)),
              ctypes.pointer(B.LossOpts(0.0, float("nan")))):
        assert lib.lce_forward_slice_ex(p, p, 0, p, 8, 8, 8, 0, 10, -100, o,
                                        p, p, p, p, p, 1 << 30, null) == 1
        assert lib.lce_forward_slice_exp_ex(p, p, 0, p, 8, 8, 8, 0, 10, -100,
                                            o, p, p, p, p, p, 1 << 30,
                                            null) == 1
        assert lib.lce_combine_slices_ex(p, p, p, p, 2, p, 8, 10, -100, o, p,
                                         p, p, 1 << 20, null) == 1
        assert lib.lce_backward_slice_ex(p, p, 0, p, p, 8, 8, 8, 0, 10, -100,
                                         o, p, 0, p, p, p, 1 << 30,
                                         null) == 1
        assert lib.lce_backward_slice_exp_ex(p, p, 0, p, p, 8, 8, 8, 0, 10,
                                             -100, o, p, p, p, p, 1 << 30,
                                             null) == 1
    for f in (lib.lce_forward_slice_ex, lib.lce_forward_slice_exp_ex):
        assert f(p, p, 0, p, 8, 8, 8, 0, 10, -100, smooth, p, p, p, null, p,
                 1 << 30, null) == 1
        assert f(p, p, 0, p, 8, 8, 8, 0, 10, -100, smooth, p, p, p, odd, p,
                 1 << 30, null) == 1
        # no smoothing: the sums are optional; a small workspace is next
        assert f(p, p, 0, p, 8, 8, 8, 0, 10, -100, zonly, p, p, p, null, p,
                 16, null) == 3
    assert lib.lce_combine_slices_ex(p, p, p, null, 2, p, 8, 10, -100,
                                     smooth, p, p, p, 1 << 20, null) == 1
    assert lib.lce_combine_slices_ex(p, p, p, odd, 2, p, 8, 10, -100,
                                     smooth, p, p, p, 1 << 20, null) == 1
    assert lib.lce_combine_slices_ex(p, p, p, null, 2, p, 8, 10, -100,
                                     zonly, p, p, p, 8, null) == 3
    assert lib.lce_backward_slice_ex(p, p, 0, p, p, 8, 8, 8, 4, 10, -100,
                                     smooth, p, 0, p, p, p, 1 << 30,
                                     null) == 1
    assert lib.lce_backward_slice_exp_ex(p, p, 0, p, p, 8, 8, 8, 0, 10, -100,
                                         smooth, p, p, p, p, 16, null) == 3
    # optional gradients: the backward wants at least one of dH, dW; the
    # scale call with neither has nothing to do
    assert lib.lce_backward(p, p, 0, p, p, 8, 8, 8, -100, p, 0, null, null, p,
                            1 << 30, null) == 1
    assert lib.lce_backward_slice(p, p, 0, p, p, 8, 8, 8, 0, 10, -100, p, 0,
                                  null, null, p, 1 << 30, null) == 1
    assert lib.lce_backward_slice_exp(p, p, 0, p, p, 8, 8, 8, 0, 10, -100, p,
                                      null, null, p, 1 << 30, null) == 1
    assert lib.lce_backward(p, p, 0, p, p, 8, 8, 8, -100, p, 0, null, p, p,
                            16, null) == 3   # dH skipped: the workspace next
    assert lib.lce_scale_gradients(null, 0, 8, 8, null, 8, p, null) == 0
    # the MLP: dWg and dWu both or neither; not every gradient left out
    assert lib.lce_mlp_backward(p, p, p, p, p, 8, 8, 64, 0, p, null, p, p, p,
                                1 << 30, null) == 1
    assert lib.lce_mlp_backward(p, p, p, p, p, 8, 8, 64, 0, null, null, null,
                                null, p, 1 << 30, null) == 1
    assert lib.lce_mlp_backward(p, p, p, p, p, 8, 8, 64, 0, p, null, null,
                                null, p, 16, null) == 3  # dx alone: valid
    assert lib.lce_scale_gradients(null, 0, 8, 8, null, 8, null, null) == 1
    # the shard combine: null or misaligned pointers
    assert lib.lce_shard_sums(null, p, p, null) == 1
    assert lib.lce_shard_sums(p, p, ctypes.c_void_p(0x1004), null) == 1
    assert lib.lce_combine_shards(p, p, null, null, p, null) == 1
    assert lib.lce_combine_shards(p, ctypes.c_void_p(0x1004), null, p, p,
                                  null) == 1
    # test hooks
    assert lib.lce_test_gemm(null, p, p, 8, 8, 8, 0, 0, null) == 1
    assert lib.lce_test_gemm(p, p, p, 8, 12, 8, 0, 0, null) == 1
    assert lib.lce_test_wait_timeout(0, null) == 1
    # the contraction variant switch is host state only
    assert lib.lce_set_cta_pair(2) == 1
    before = lib.lce_get_cta_pair()
    assert lib.lce_set_cta_pair(1) == 0 and lib.lce_get_cta_pair() == 1
    assert lib.lce_set_cta_pair(0) == 0 and lib.lce_get_cta_pair() == 0
    assert lib.lce_set_cta_pair(before) == 0
    assert lib.lce_set_wave_sync(2) == 1
    before = lib.lce_get_wave_sync()
    assert lib.lce_set_wave_sync(0) == 0 and lib.lce_get_wave_sync() == 0
    assert lib.lce_set_wave_sync(1) == 0 and lib.lce_get_wave_sync() == 1
    assert lib.lce_set_wave_sync(before) == 0


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    from chunked_lm_head_gemm_gb300 import _binding as B
    from chunked_lm_head_gemm_gb300 import build as Bld
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(Bld, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        B.load()
