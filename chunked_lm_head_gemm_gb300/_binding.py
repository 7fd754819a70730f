"""ctypes binding of liblce.so (include/lce.h): argument marshalling only.

Every step of the loss runs in the library's CUDA kernels; this module only
checks tensors, passes their device pointers and the current CUDA stream,
and raises on a non-OK status. There is no fallback: if the library is not
built or the device is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lib = None
_lock = threading.Lock()

LCE_OK = 0
LCE_ERR_INVALID_ARG = 1
LCE_ERR_UNSUPPORTED = 2
LCE_ERR_WORKSPACE = 3
LCE_ERR_LABEL_RANGE = 4
LCE_ERR_TIMEOUT = 5
LCE_ERR_CUDA = 6

LCE_BF16 = 0
LCE_F32 = 1

IGNORE_INDEX = -100

EXPORTED = ("lce_workspace_size", "lce_default_chunk_rows", "lce_forward",
            "lce_backward", "lce_get_error", "lce_status_string",
            "lce_last_cuda_error", "lce_test_gemm", "lce_test_wait_timeout",
            "lce_profile_start", "lce_profile_stop", "lce_forward_static",
            "lce_forward_backward", "lce_scale_gradients",
            "lce_set_cta_pair", "lce_get_cta_pair", "lce_mlp_workspace_size",
            "lce_mlp_forward", "lce_mlp_backward", "lce_count_valid",
            "lce_forward_slice", "lce_combine_workspace_size",
            "lce_combine_slices", "lce_backward_slice", "lce_set_wave_sync",
            "lce_get_wave_sync", "lce_slice_exp_workspace_size",
            "lce_forward_slice_exp", "lce_backward_slice_exp",
            "lce_forward_ex", "lce_backward_ex", "lce_forward_backward_ex",
            "lce_shard_sums", "lce_combine_shards", "lce_forward_slice_ex",
            "lce_combine_slices_ex", "lce_backward_slice_ex",
            "lce_forward_slice_exp_ex", "lce_backward_slice_exp_ex")

KERNEL_KINDS = 22


class LossOpts(ctypes.Structure):
    """lce_loss_opts: label smoothing in [0, 1] and the z-loss coefficient."""
    _fields_ = [("label_smoothing", ctypes.c_float),
                ("z_loss", ctypes.c_float)]


class KernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double), ("flops", ctypes.c_double)]


class LCEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        lib = _lib
        name = lib.lce_status_string(status).decode() if lib else str(status)
        detail = lib.lce_last_cuda_error().decode() if lib else ""
        super().__init__(f"{where}: {name}" + (f" ({detail})" if detail else ""))


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False):
    """Open liblce.so and declare the C signatures. Raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"CUDA library not built: {path} is missing "
                    "(run __graft_entry__.build() or python -m "
                    "chunked_lm_head_gemm_gb300.build)")
            _build.build()
        lib = ctypes.CDLL(path)
        p, i64, i32, u64, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                ctypes.c_uint64, ctypes.c_size_t)
        lib.lce_workspace_size.argtypes = [i64, i64, i64, i32, i64]
        lib.lce_workspace_size.restype = sz
        lib.lce_default_chunk_rows.argtypes = [i64, i64, i64]
        lib.lce_default_chunk_rows.restype = i64
        lib.lce_forward.argtypes = [p, p, i32, p, i64, i64, i64, i64, p, p, p,
                                    sz, p]
        lib.lce_forward.restype = i32
        lib.lce_backward.argtypes = [p, p, i32, p, p, i64, i64, i64, i64, p,
                                     i64, p, p, p, sz, p]
        lib.lce_backward.restype = i32
        lib.lce_get_error.argtypes = [p]
        lib.lce_get_error.restype = i32
        lib.lce_status_string.argtypes = [i32]
        lib.lce_status_string.restype = ctypes.c_char_p
        lib.lce_last_cuda_error.argtypes = []
        lib.lce_last_cuda_error.restype = ctypes.c_char_p
        lib.lce_test_gemm.argtypes = [p, p, p, i64, i64, i64, i32, i32, p]
        lib.lce_test_gemm.restype = i32
        lib.lce_test_wait_timeout.argtypes = [u64, p]
        lib.lce_test_wait_timeout.restype = i32
        lib.lce_forward_backward.argtypes = [p, p, i32, p, i64, i64, i64, i64,
                                             i64, p, p, p, p, p, sz, p]
        lib.lce_forward_backward.restype = i32
        opts = ctypes.POINTER(LossOpts)
        lib.lce_forward_ex.argtypes = [p, p, i32, p, i64, i64, i64, i64, opts,
                                       p, p, p, sz, p]
        lib.lce_forward_ex.restype = i32
        lib.lce_backward_ex.argtypes = [p, p, i32, p, p, i64, i64, i64, i64,
                                        opts, p, i64, p, p, p, sz, p]
        lib.lce_backward_ex.restype = i32
        lib.lce_forward_backward_ex.argtypes = [p, p, i32, p, i64, i64, i64,
                                                i64, opts, i64, p, p, p, p, p,
                                                sz, p]
        lib.lce_forward_backward_ex.restype = i32
        lib.lce_shard_sums.argtypes = [p, p, p, p]
        lib.lce_shard_sums.restype = i32
        lib.lce_combine_shards.argtypes = [p, p, p, p, p, p]
        lib.lce_combine_shards.restype = i32
        lib.lce_scale_gradients.argtypes = [p, i32, i64, i64, p, i64, p, p]
        lib.lce_scale_gradients.restype = i32
        lib.lce_count_valid.argtypes = [p, i64, i64, i64, p, p]
        lib.lce_count_valid.restype = i32
        lib.lce_forward_slice.argtypes = [p, p, i32, p, i64, i64, i64, i64,
                                          i64, i64, p, p, p, p, sz, p]
        lib.lce_forward_slice.restype = i32
        lib.lce_combine_workspace_size.argtypes = [i64]
        lib.lce_combine_workspace_size.restype = sz
        lib.lce_combine_slices.argtypes = [p, p, p, i64, p, i64, i64, i64, p,
                                           p, p, sz, p]
        lib.lce_combine_slices.restype = i32
        lib.lce_backward_slice.argtypes = [p, p, i32, p, p, i64, i64, i64,
                                           i64, i64, i64, p, i64, p, p, p, sz,
                                           p]
        lib.lce_backward_slice.restype = i32
        lib.lce_slice_exp_workspace_size.argtypes = [i64, i64, i64, i32]
        lib.lce_slice_exp_workspace_size.restype = sz
        lib.lce_forward_slice_exp.argtypes = [p, p, i32, p, i64, i64, i64,
                                              i64, i64, i64, p, p, p, p, sz,
                                              p]
        lib.lce_forward_slice_exp.restype = i32
        lib.lce_backward_slice_exp.argtypes = [p, p, i32, p, p, i64, i64, i64,
                                               i64, i64, i64, p, p, p, p, sz,
                                               p]
        lib.lce_backward_slice_exp.restype = i32
        lib.lce_forward_slice_ex.argtypes = [p, p, i32, p, i64, i64, i64,
                                             i64, i64, i64, opts, p, p, p, p,
                                             p, sz, p]
        lib.lce_forward_slice_ex.restype = i32
        lib.lce_combine_slices_ex.argtypes = [p, p, p, p, i64, p, i64, i64,
                                              i64, opts, p, p, p, sz, p]
        lib.lce_combine_slices_ex.restype = i32
        lib.lce_backward_slice_ex.argtypes = [p, p, i32, p, p, i64, i64, i64,
                                              i64, i64, i64, opts, p, i64, p,
                                              p, p, sz, p]
        lib.lce_backward_slice_ex.restype = i32
        lib.lce_forward_slice_exp_ex.argtypes = [p, p, i32, p, i64, i64, i64,
                                                 i64, i64, i64, opts, p, p, p,
                                                 p, p, sz, p]
        lib.lce_forward_slice_exp_ex.restype = i32
        lib.lce_backward_slice_exp_ex.argtypes = [p, p, i32, p, p, i64, i64,
                                                  i64, i64, i64, i64, opts, p,
                                                  p, p, p, sz, p]
        lib.lce_backward_slice_exp_ex.restype = i32
        lib.lce_mlp_workspace_size.argtypes = [i64, i64, i64, i64]
        lib.lce_mlp_workspace_size.restype = sz
        lib.lce_mlp_forward.argtypes = [p, p, p, p, i64, i64, i64, i64, p, p,
                                        sz, p]
        lib.lce_mlp_forward.restype = i32
        lib.lce_mlp_backward.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p,
                                         p, p, p, p, sz, p]
        lib.lce_mlp_backward.restype = i32
        lib.lce_set_cta_pair.argtypes = [i32]
        lib.lce_set_cta_pair.restype = i32
        lib.lce_get_cta_pair.argtypes = []
        lib.lce_get_cta_pair.restype = i32
        lib.lce_set_wave_sync.argtypes = [i32]
        lib.lce_set_wave_sync.restype = i32
        lib.lce_get_wave_sync.argtypes = []
        lib.lce_get_wave_sync.restype = i32
        lib.lce_forward_static.argtypes = [p, p, p, i64, i64, i64, i64, p, p,
                                           p]
        lib.lce_forward_static.restype = i32
        lib.lce_profile_start.argtypes = []
        lib.lce_profile_start.restype = i32
        lib.lce_profile_stop.argtypes = [ctypes.POINTER(KernelStat)]
        lib.lce_profile_stop.restype = i32
        _lib = lib
        return lib


def _check(status: int, where: str):
    if status != LCE_OK:
        raise LCEError(status, where)


def _stream_ptr(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return LCE_BF16
    if t.dtype == torch.float32:
        return LCE_F32
    raise TypeError(f"unsupported dtype {t.dtype}; use bfloat16 or float32")


def _check_inputs(h, W, labels):
    if not (h.is_cuda and W.is_cuda and labels.is_cuda):
        raise ValueError("h, W and labels must be CUDA tensors")
    if h.dim() != 2 or W.dim() != 2 or labels.dim() != 1:
        raise ValueError("expected h [L,H], W [V,H], labels [L]")
    if h.shape[1] != W.shape[1] or labels.shape[0] != h.shape[0]:
        raise ValueError(f"shape mismatch: h {tuple(h.shape)}, W "
                         f"{tuple(W.shape)}, labels {tuple(labels.shape)}")
    if h.dtype != W.dtype:
        raise TypeError("h and W must have the same dtype")
    if labels.dtype != torch.int64:
        raise TypeError("labels must be int64")
    if not (h.is_contiguous() and W.is_contiguous() and labels.is_contiguous()):
        raise ValueError("h, W and labels must be contiguous")


def workspace_size(L: int, H: int, V: int, dtype=torch.bfloat16,
                   chunk_rows: int = 0) -> int:
    code = LCE_BF16 if dtype == torch.bfloat16 else LCE_F32
    n = load().lce_workspace_size(L, H, V, code, chunk_rows)
    if n == 0:
        raise ValueError(f"invalid sizes L={L} H={H} V={V} chunk={chunk_rows}")
    return n


def default_chunk_rows(L: int, H: int, V: int) -> int:
    return load().lce_default_chunk_rows(L, H, V)


def alloc_workspace(L, H, V, dtype, chunk_rows, device) -> torch.Tensor:
    return torch.empty(workspace_size(L, H, V, dtype, chunk_rows),
                       dtype=torch.uint8, device=device)


def _opts(label_smoothing: float, z_loss: float):
    """The lce_loss_opts pointer for a loss variant, or None (plain loss)."""
    if label_smoothing == 0.0 and z_loss == 0.0:
        return None
    return ctypes.pointer(LossOpts(float(label_smoothing), float(z_loss)))


def forward(h: torch.Tensor, W: torch.Tensor, labels: torch.Tensor,
            ignore_index: int = IGNORE_INDEX, workspace=None,
            loss_out=None, lse_out=None, label_smoothing: float = 0.0,
            z_loss: float = 0.0):
    """Returns (loss [scalar fp32], lse [L] fp32), both on h's device.
    label_smoothing / z_loss select a loss variant (lce_forward_ex)."""
    lib = load()
    _check_inputs(h, W, labels)
    L, H = h.shape
    V = W.shape[0]
    dev = h.device
    if workspace is None:
        workspace = alloc_workspace(L, H, V, h.dtype, 0, dev)
    loss = loss_out if loss_out is not None else torch.empty((), dtype=torch.float32, device=dev)
    lse = lse_out if lse_out is not None else torch.empty(L, dtype=torch.float32, device=dev)
    opts = _opts(label_smoothing, z_loss)
    if opts is None:
        st = lib.lce_forward(h.data_ptr(), W.data_ptr(), _dtype_code(h),
                             labels.data_ptr(), L, H, V, ignore_index,
                             loss.data_ptr(), lse.data_ptr(),
                             workspace.data_ptr(), workspace.numel(),
                             _stream_ptr(dev))
        _check(st, "lce_forward")
    else:
        st = lib.lce_forward_ex(h.data_ptr(), W.data_ptr(), _dtype_code(h),
                                labels.data_ptr(), L, H, V, ignore_index,
                                opts, loss.data_ptr(), lse.data_ptr(),
                                workspace.data_ptr(), workspace.numel(),
                                _stream_ptr(dev))
        _check(st, "lce_forward_ex")
    return loss, lse


def backward(h: torch.Tensor, W: torch.Tensor, labels: torch.Tensor,
             lse: torch.Tensor, dloss: torch.Tensor,
             ignore_index: int = IGNORE_INDEX, chunk_rows: int = 0,
             workspace=None, dH_out=None, dW_out=None,
             label_smoothing: float = 0.0, z_loss: float = 0.0,
             compute_dH: bool = True, compute_dW: bool = True):
    """Returns (dH [L,H] of h's dtype, dW [V,H] fp32). The loss variant
    must be the forward's. compute_dH / compute_dW = False skips that
    gradient's contraction (returned as None; at least one is needed)."""
    lib = load()
    _check_inputs(h, W, labels)
    L, H = h.shape
    V = W.shape[0]
    dev = h.device
    if lse.dtype != torch.float32 or lse.shape != (L,) or not lse.is_cuda:
        raise ValueError("lse must be a CUDA float32 [L] tensor")
    dloss = dloss.reshape(1).to(device=dev, dtype=torch.float32).contiguous()
    if workspace is None:
        workspace = alloc_workspace(L, H, V, h.dtype, chunk_rows, dev)
    dH, dW = _grad_outputs(h, V, dH_out, dW_out, compute_dH, compute_dW)
    opts = _opts(label_smoothing, z_loss)
    if opts is None:
        st = lib.lce_backward(h.data_ptr(), W.data_ptr(), _dtype_code(h),
                              labels.data_ptr(), lse.data_ptr(), L, H, V,
                              ignore_index, dloss.data_ptr(), chunk_rows,
                              _ptr(dH), _ptr(dW), workspace.data_ptr(),
                              workspace.numel(), _stream_ptr(dev))
        _check(st, "lce_backward")
    else:
        st = lib.lce_backward_ex(h.data_ptr(), W.data_ptr(), _dtype_code(h),
                                 labels.data_ptr(), lse.data_ptr(), L, H, V,
                                 ignore_index, opts, dloss.data_ptr(),
                                 chunk_rows, _ptr(dH), _ptr(dW),
                                 workspace.data_ptr(), workspace.numel(),
                                 _stream_ptr(dev))
        _check(st, "lce_backward_ex")
    return dH, dW


def _ptr(t):
    """A tensor's device pointer, or None (NULL) for an absent one."""
    return None if t is None else t.data_ptr()


def _grad_outputs(h, V, dH_out, dW_out, compute_dH, compute_dW):
    """The dH [L,H] (h's dtype) and dW [V,H] fp32 outputs, None where the
    gradient is not wanted."""
    L, H = h.shape
    dH = dW = None
    if compute_dH:
        dH = dH_out if dH_out is not None else torch.empty_like(h)
    if compute_dW:
        dW = dW_out if dW_out is not None else torch.empty(
            V, H, dtype=torch.float32, device=h.device)
    return dH, dW


def forward_backward(h: torch.Tensor, W: torch.Tensor, labels: torch.Tensor,
                     ignore_index: int = IGNORE_INDEX, chunk_rows: int = 0,
                     workspace=None, loss_out=None, lse_out=None, dH_out=None,
                     dW_out=None, label_smoothing: float = 0.0,
                     z_loss: float = 0.0, compute_dH: bool = True,
                     compute_dW: bool = True):
    """Loss, lse and the gradients of the loss itself (dloss = 1) in one
    call, without recomputing the logits. Returns (loss, lse, dH, dW);
    compute_dH / compute_dW = False skips that gradient (None)."""
    lib = load()
    _check_inputs(h, W, labels)
    L, H = h.shape
    V = W.shape[0]
    dev = h.device
    if workspace is None:
        workspace = alloc_workspace(L, H, V, h.dtype, chunk_rows, dev)
    loss = loss_out if loss_out is not None else torch.empty((), dtype=torch.float32, device=dev)
    lse = lse_out if lse_out is not None else torch.empty(L, dtype=torch.float32, device=dev)
    dH, dW = _grad_outputs(h, V, dH_out, dW_out, compute_dH, compute_dW)
    opts = _opts(label_smoothing, z_loss)
    if opts is None:
        st = lib.lce_forward_backward(h.data_ptr(), W.data_ptr(),
                                      _dtype_code(h), labels.data_ptr(), L, H,
                                      V, ignore_index, chunk_rows,
                                      loss.data_ptr(), lse.data_ptr(),
                                      _ptr(dH), _ptr(dW),
                                      workspace.data_ptr(), workspace.numel(),
                                      _stream_ptr(dev))
        _check(st, "lce_forward_backward")
    else:
        st = lib.lce_forward_backward_ex(h.data_ptr(), W.data_ptr(),
                                         _dtype_code(h), labels.data_ptr(), L,
                                         H, V, ignore_index, opts, chunk_rows,
                                         loss.data_ptr(), lse.data_ptr(),
                                         _ptr(dH), _ptr(dW),
                                         workspace.data_ptr(),
                                         workspace.numel(), _stream_ptr(dev))
        _check(st, "lce_forward_backward_ex")
    return loss, lse, dH, dW


def scale_gradients(dH, dW, dloss: torch.Tensor):
    """dH *= dloss and dW *= dloss in place (dloss a device scalar); either
    gradient may be None."""
    ref = dH if dH is not None else dW
    if ref is None:
        return dH, dW
    L, H = dH.shape if dH is not None else (1, dW.shape[1])
    V = dW.shape[0] if dW is not None else 1
    code = _dtype_code(dH) if dH is not None else LCE_BF16
    dloss = dloss.reshape(1).to(device=ref.device,
                                dtype=torch.float32).contiguous()
    st = load().lce_scale_gradients(_ptr(dH), code, L, H, _ptr(dW), V,
                                    dloss.data_ptr(), _stream_ptr(ref.device))
    _check(st, "lce_scale_gradients")
    return dH, dW


def count_valid(labels: torch.Tensor, V: int,
                ignore_index: int = IGNORE_INDEX, out=None) -> torch.Tensor:
    """Device int64 [1]: rows whose label is not ignore_index and lies in
    [0, V) (the N of the mean loss); no host synchronisation."""
    if labels.dtype != torch.int64 or labels.dim() != 1 or not labels.is_cuda:
        raise ValueError("labels must be a 1-D int64 CUDA tensor")
    labels = labels.contiguous()
    if out is None:
        out = torch.empty(1, dtype=torch.int64, device=labels.device)
    st = load().lce_count_valid(labels.data_ptr(), labels.numel(), V,
                                ignore_index, out.data_ptr(),
                                _stream_ptr(labels.device))
    _check(st, "lce_count_valid")
    return out


def shard_sums(loss_local: torch.Tensor, n_local: torch.Tensor,
               out=None) -> torch.Tensor:
    """Device float64 [2] = (N_r loss_r, N_r) of one row shard, to be summed
    over the shards (lce_shard_sums)."""
    loss_local = loss_local.reshape(1).to(torch.float32).contiguous()
    n_local = n_local.reshape(1).to(torch.int64).contiguous()
    dev = loss_local.device
    if out is None:
        out = torch.empty(2, dtype=torch.float64, device=dev)
    st = load().lce_shard_sums(loss_local.data_ptr(), n_local.data_ptr(),
                               out.data_ptr(), _stream_ptr(dev))
    _check(st, "lce_shard_sums")
    return out


def combine_shards(sums: torch.Tensor, n_local: torch.Tensor,
                   dloss: torch.Tensor | None = None):
    """From the shards' summed (S, N): (loss = S / N, this shard's gradient
    weight dloss N_r / N), device float32 scalars, 0 when N = 0
    (lce_combine_shards)."""
    if sums.dtype != torch.float64 or sums.numel() != 2 or not sums.is_cuda:
        raise ValueError("sums must be a CUDA float64 tensor of 2 elements")
    sums = sums.contiguous()
    dev = sums.device
    n_local = n_local.reshape(1).to(torch.int64).contiguous()
    d = None
    if dloss is not None:
        d = dloss.reshape(1).to(device=dev, dtype=torch.float32).contiguous()
    loss = torch.empty((), dtype=torch.float32, device=dev)
    weight = torch.empty((), dtype=torch.float32, device=dev)
    st = load().lce_combine_shards(sums.data_ptr(), n_local.data_ptr(),
                                   d.data_ptr() if d is not None else None,
                                   loss.data_ptr(), weight.data_ptr(),
                                   _stream_ptr(dev))
    _check(st, "lce_combine_shards")
    return loss, weight


def _slice_out(out, L, label_smoothing, dev):
    """Rows m, s, zy (and zsum under label smoothing) of a [3 or 4, L]
    float32 tensor."""
    rows = 4 if label_smoothing != 0.0 else 3
    if out is None:
        out = torch.empty(rows, L, dtype=torch.float32, device=dev)
    if out.dtype != torch.float32 or out.shape != (rows, L):
        raise ValueError(f"out must be float32 [{rows}, {L}]")
    return out, tuple(out[r] for r in range(rows))


def forward_slice(h: torch.Tensor, W_slice: torch.Tensor,
                  labels: torch.Tensor, v0: int, V_total: int,
                  ignore_index: int = IGNORE_INDEX, workspace=None,
                  out=None, label_smoothing: float = 0.0,
                  z_loss: float = 0.0):
    """One vocabulary slice (W_slice = rows v0 .. v0 + Vs - 1 of the head):
    returns (m, s, zy), each float32 [L]: the slice's per-row max logit, sum
    of exp(z - m), and label logit (0 where the label is elsewhere); under
    label smoothing also zsum, the slice's per-row sum of logits, as a
    fourth (lce_forward_slice_ex)."""
    lib = load()
    _check_inputs(h, W_slice, labels)
    L, H = h.shape
    Vs = W_slice.shape[0]
    dev = h.device
    if workspace is None:
        workspace = alloc_workspace(L, H, Vs, h.dtype, 0, dev)
    out, rows = _slice_out(out, L, label_smoothing, dev)
    opts = _opts(label_smoothing, z_loss)
    if opts is None:
        st = lib.lce_forward_slice(h.data_ptr(), W_slice.data_ptr(),
                                   _dtype_code(h), labels.data_ptr(), L, H,
                                   Vs, v0, V_total, ignore_index,
                                   rows[0].data_ptr(), rows[1].data_ptr(),
                                   rows[2].data_ptr(), workspace.data_ptr(),
                                   workspace.numel(), _stream_ptr(dev))
    else:
        st = lib.lce_forward_slice_ex(
            h.data_ptr(), W_slice.data_ptr(), _dtype_code(h),
            labels.data_ptr(), L, H, Vs, v0, V_total, ignore_index, opts,
            rows[0].data_ptr(), rows[1].data_ptr(), rows[2].data_ptr(),
            rows[3].data_ptr() if len(rows) == 4 else None,
            workspace.data_ptr(), workspace.numel(), _stream_ptr(dev))
    _check(st, "lce_forward_slice")
    return rows


def combine_slices(m: torch.Tensor, s: torch.Tensor, zy: torch.Tensor,
                   labels: torch.Tensor, V_total: int,
                   ignore_index: int = IGNORE_INDEX, workspace=None,
                   zsum=None, label_smoothing: float = 0.0,
                   z_loss: float = 0.0):
    """m, s, zy (and zsum under label smoothing): float32 [P, L] (every
    slice's forward_slice output, in the same slice order on every
    process). Returns (loss, lse [L])."""
    lib = load()
    P, L = m.shape
    ts = (m, s, zy) if zsum is None else (m, s, zy, zsum)
    for t in ts:
        if t.dtype != torch.float32 or t.shape != (P, L) or not t.is_cuda:
            raise ValueError("m, s, zy, zsum must be CUDA float32 [P, L] "
                             "tensors")
    m, s, zy = m.contiguous(), s.contiguous(), zy.contiguous()
    zsum = zsum.contiguous() if zsum is not None else None
    labels = labels.contiguous()
    dev = m.device
    if workspace is None:
        workspace = torch.empty(lib.lce_combine_workspace_size(L),
                                dtype=torch.uint8, device=dev)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    lse = torch.empty(L, dtype=torch.float32, device=dev)
    opts = _opts(label_smoothing, z_loss)
    if opts is None:
        st = lib.lce_combine_slices(m.data_ptr(), s.data_ptr(), zy.data_ptr(),
                                    P, labels.data_ptr(), L, V_total,
                                    ignore_index, loss.data_ptr(),
                                    lse.data_ptr(), workspace.data_ptr(),
                                    workspace.numel(), _stream_ptr(dev))
    else:
        st = lib.lce_combine_slices_ex(
            m.data_ptr(), s.data_ptr(), zy.data_ptr(),
            zsum.data_ptr() if zsum is not None else None, P,
            labels.data_ptr(), L, V_total, ignore_index, opts,
            loss.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
            workspace.numel(), _stream_ptr(dev))
    _check(st, "lce_combine_slices")
    return loss, lse


def backward_slice(h: torch.Tensor, W_slice: torch.Tensor,
                   labels: torch.Tensor, lse: torch.Tensor,
                   dloss: torch.Tensor, v0: int, V_total: int,
                   ignore_index: int = IGNORE_INDEX, chunk_rows: int = 0,
                   workspace=None, label_smoothing: float = 0.0,
                   z_loss: float = 0.0, compute_dH: bool = True,
                   compute_dW: bool = True):
    """One vocabulary slice's backward from the merged lse: returns
    (dH_part [L,H] float32, whose sum over slices is dH; dW_slice [Vs,H]);
    compute_dH / compute_dW = False skips that one (None)."""
    lib = load()
    _check_inputs(h, W_slice, labels)
    L, H = h.shape
    Vs = W_slice.shape[0]
    dev = h.device
    if lse.dtype != torch.float32 or lse.shape != (L,) or not lse.is_cuda:
        raise ValueError("lse must be a CUDA float32 [L] tensor")
    dloss = dloss.reshape(1).to(device=dev, dtype=torch.float32).contiguous()
    if workspace is None:
        workspace = alloc_workspace(L, H, Vs, h.dtype, chunk_rows, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    dH = torch.empty(L, H, **f32) if compute_dH else None
    dW = torch.empty(Vs, H, **f32) if compute_dW else None
    st = lib.lce_backward_slice_ex(h.data_ptr(), W_slice.data_ptr(),
                                   _dtype_code(h), labels.data_ptr(),
                                   lse.data_ptr(), L, H, Vs, v0, V_total,
                                   ignore_index,
                                   _opts(label_smoothing, z_loss),
                                   dloss.data_ptr(), chunk_rows,
                                   _ptr(dH), _ptr(dW),
                                   workspace.data_ptr(), workspace.numel(),
                                   _stream_ptr(dev))
    _check(st, "lce_backward_slice")
    return dH, dW


def slice_exp_workspace(L: int, H: int, Vs: int, dtype, device):
    """The workspace forward_slice_exp fills and backward_slice_exp reads."""
    n = load().lce_slice_exp_workspace_size(
        L, H, Vs, LCE_F32 if dtype == torch.float32 else LCE_BF16)
    if n == 0:
        raise ValueError("invalid sizes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def forward_slice_exp(h, W_slice, labels, v0: int, V_total: int, workspace,
                      ignore_index: int = IGNORE_INDEX, out=None,
                      label_smoothing: float = 0.0, z_loss: float = 0.0):
    """forward_slice that also keeps the slice's tile exponentials in
    `workspace` (from slice_exp_workspace) for backward_slice_exp."""
    lib = load()
    _check_inputs(h, W_slice, labels)
    L, H = h.shape
    Vs = W_slice.shape[0]
    out, rows = _slice_out(out, L, label_smoothing, h.device)
    st = lib.lce_forward_slice_exp_ex(
        h.data_ptr(), W_slice.data_ptr(), _dtype_code(h), labels.data_ptr(),
        L, H, Vs, v0, V_total, ignore_index, _opts(label_smoothing, z_loss),
        rows[0].data_ptr(), rows[1].data_ptr(), rows[2].data_ptr(),
        rows[3].data_ptr() if len(rows) == 4 else None,
        workspace.data_ptr(), workspace.numel(), _stream_ptr(h.device))
    _check(st, "lce_forward_slice_exp")
    return rows


def backward_slice_exp(h, W_slice, labels, lse, dloss, v0: int, V_total: int,
                       workspace, ignore_index: int = IGNORE_INDEX,
                       label_smoothing: float = 0.0, z_loss: float = 0.0,
                       compute_dH: bool = True, compute_dW: bool = True):
    """The slice's backward from the exponentials forward_slice_exp kept:
    returns (dH_part [L,H] float32, dW_slice [Vs,H] float32), None for a
    gradient not asked for."""
    lib = load()
    _check_inputs(h, W_slice, labels)
    L, H = h.shape
    Vs = W_slice.shape[0]
    dev = h.device
    if lse.dtype != torch.float32 or lse.shape != (L,) or not lse.is_cuda:
        raise ValueError("lse must be a CUDA float32 [L] tensor")
    dloss = dloss.reshape(1).to(device=dev, dtype=torch.float32).contiguous()
    f32 = dict(dtype=torch.float32, device=dev)
    dH = torch.empty(L, H, **f32) if compute_dH else None
    dW = torch.empty(Vs, H, **f32) if compute_dW else None
    st = lib.lce_backward_slice_exp_ex(h.data_ptr(), W_slice.data_ptr(),
                                       _dtype_code(h), labels.data_ptr(),
                                       lse.data_ptr(), L, H, Vs, v0, V_total,
                                       ignore_index,
                                       _opts(label_smoothing, z_loss),
                                       dloss.data_ptr(), _ptr(dH), _ptr(dW),
                                       workspace.data_ptr(),
                                       workspace.numel(),
                                       _stream_ptr(dev))
    _check(st, "lce_backward_slice_exp")
    return dH, dW


def get_error(device=None) -> int:
    """Synchronises the current stream and returns (and clears) the device
    error status: LCE_OK, LCE_ERR_LABEL_RANGE or LCE_ERR_TIMEOUT."""
    return load().lce_get_error(_stream_ptr(device))


def tc_gemm(A: torch.Tensor, B: torch.Tensor, M: int, N: int, K: int,
              a_mn: bool, b_mn: bool) -> torch.Tensor:
    """D = A B (fp32) through the tensor-core building block.
    A: [M,K] if not a_mn else [K,M]; B: [N,K] if not b_mn else [K,N]."""
    lib = load()
    D = torch.empty(M, N, dtype=torch.float32, device=A.device)
    st = lib.lce_test_gemm(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K,
                           int(a_mn), int(b_mn), _stream_ptr(A.device))
    _check(st, "lce_test_gemm")
    return D


def wait_timeout_probe(timeout_ns: int, device=None):
    st = load().lce_test_wait_timeout(timeout_ns, _stream_ptr(device))
    _check(st, "lce_test_wait_timeout")


def _check_mlp(x, Wg, Wu, Wd):
    ts = (x, Wg, Wu, Wd)
    if not all(t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()
               for t in ts):
        raise ValueError("x, Wg, Wu, Wd must be contiguous bf16 CUDA tensors")
    L, H = x.shape
    I = Wg.shape[0]
    if Wg.shape != (I, H) or Wu.shape != (I, H) or Wd.shape != (H, I):
        raise ValueError(f"shape mismatch: x {tuple(x.shape)}, Wg "
                         f"{tuple(Wg.shape)}, Wu {tuple(Wu.shape)}, Wd "
                         f"{tuple(Wd.shape)}")
    return L, H, I


def mlp_workspace_size(L: int, H: int, I: int, chunk_rows: int = 0) -> int:
    n = load().lce_mlp_workspace_size(L, H, I, chunk_rows)
    if n == 0:
        raise ValueError(f"invalid MLP sizes L={L} H={H} I={I}")
    return n


def mlp_forward(x, Wg, Wu, Wd, chunk_rows: int = 0, workspace=None,
                y_out=None):
    """y = (silu(x Wg^T) * (x Wu^T)) Wd^T over row chunks (bf16)."""
    lib = load()
    L, H, I = _check_mlp(x, Wg, Wu, Wd)
    if workspace is None:
        workspace = torch.empty(mlp_workspace_size(L, H, I, chunk_rows),
                                dtype=torch.uint8, device=x.device)
    y = y_out if y_out is not None else torch.empty_like(x)
    st = lib.lce_mlp_forward(x.data_ptr(), Wg.data_ptr(), Wu.data_ptr(),
                             Wd.data_ptr(), L, H, I, chunk_rows, y.data_ptr(),
                             workspace.data_ptr(), workspace.numel(),
                             _stream_ptr(x.device))
    _check(st, "lce_mlp_forward")
    return y


def mlp_backward(x, Wg, Wu, Wd, dy, chunk_rows: int = 0, workspace=None,
                 dx_out=None, dWg_out=None, dWu_out=None, dWd_out=None,
                 compute_dx: bool = True, compute_dWgu: bool = True,
                 compute_dWd: bool = True):
    """Returns (dx bf16 [L,H], dWg fp32 [I,H], dWu fp32 [I,H], dWd fp32
    [H,I]) for upstream gradient dy, recomputing the chunk intermediates.
    compute_dx / compute_dWgu (dWg and dWu) / compute_dWd = False skips
    that gradient's contraction (returned as None)."""
    lib = load()
    L, H, I = _check_mlp(x, Wg, Wu, Wd)
    if not (dy.is_cuda and dy.dtype == torch.bfloat16 and dy.is_contiguous()
            and dy.shape == (L, H)):
        raise ValueError("dy must be a contiguous bf16 CUDA [L,H] tensor")
    dev = x.device
    if workspace is None:
        workspace = torch.empty(mlp_workspace_size(L, H, I, chunk_rows),
                                dtype=torch.uint8, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    dx = dWg = dWu = dWd = None
    if compute_dx:
        dx = dx_out if dx_out is not None else torch.empty_like(x)
    if compute_dWgu:
        dWg = dWg_out if dWg_out is not None else torch.empty(I, H, **f32)
        dWu = dWu_out if dWu_out is not None else torch.empty(I, H, **f32)
    if compute_dWd:
        dWd = dWd_out if dWd_out is not None else torch.empty(H, I, **f32)
    st = lib.lce_mlp_backward(x.data_ptr(), Wg.data_ptr(), Wu.data_ptr(),
                              Wd.data_ptr(), dy.data_ptr(), L, H, I,
                              chunk_rows, _ptr(dx), _ptr(dWg), _ptr(dWu),
                              _ptr(dWd), workspace.data_ptr(),
                              workspace.numel(), _stream_ptr(dev))
    _check(st, "lce_mlp_backward")
    return dx, dWg, dWu, dWd


def set_cta_pair(enable: bool):
    """Run the contractions on CTA pairs (cta_group::2) or single CTAs."""
    _check(load().lce_set_cta_pair(1 if enable else 0), "lce_set_cta_pair")


def get_cta_pair() -> bool:
    return bool(load().lce_get_cta_pair())


def set_wave_sync(enable: bool):
    """Wave pacing of the contractions on (default) or off; same results."""
    _check(load().lce_set_wave_sync(1 if enable else 0), "lce_set_wave_sync")


def get_wave_sync() -> bool:
    return bool(load().lce_get_wave_sync())


def profile_start():
    """Time every kernel this thread launches through the library."""
    _check(load().lce_profile_start(), "lce_profile_start")


def profile_stop() -> dict:
    """Waits for the recorded launches; returns {kind: (launches, total_ms,
    flops)} for the kinds that ran."""
    arr = (KernelStat * KERNEL_KINDS)()
    _check(load().lce_profile_stop(arr), "lce_profile_stop")
    return {a.name.decode(): (a.launches, a.total_ms, a.flops) for a in arr
            if a.launches}


class LinearCrossEntropy(torch.autograd.Function):
    """loss = mean cross entropy of h W^T against labels, without the logits.

    fused=False: forward saves only lse [L] (4 bytes per row); backward
    recomputes the logits chunk by chunk in the library.
    fused=True: forward computes the loss and the gradients in one call
    (no recompute) and keeps dH, dW (for dloss = 1) until backward, which
    returns copies scaled by dloss. The kept tensors are never modified, so
    a retained graph gives the same gradients again; the cost is memory:
    dH and dW (L H + 4 V H bytes for bf16 h) stay allocated from the forward
    until the graph is freed, and backward briefly holds the scaled copies
    as well."""

    @staticmethod
    def forward(ctx, h, W, labels, ignore_index=IGNORE_INDEX, chunk_rows=0,
                fused=False, label_smoothing=0.0, z_loss=0.0):
        ctx.ignore_index = ignore_index
        ctx.chunk_rows = chunk_rows
        ctx.fused = fused
        ctx.w_dtype = W.dtype
        ctx.variant = dict(label_smoothing=label_smoothing, z_loss=z_loss)
        # only the gradients autograd asks for are computed (a frozen head:
        # no dW contraction)
        ctx.want = dict(compute_dH=ctx.needs_input_grad[0],
                        compute_dW=ctx.needs_input_grad[1])
        if fused and any(ctx.want.values()):
            loss, _, dH, dW = forward_backward(h, W, labels, ignore_index,
                                               chunk_rows, **ctx.variant,
                                               **ctx.want)
            ctx.save_for_backward(dH, dW)
        else:
            ctx.fused = False
            loss, lse = forward(h, W, labels, ignore_index, **ctx.variant)
            ctx.save_for_backward(h, W, labels, lse)
        return loss

    @staticmethod
    def backward(ctx, dloss):
        if not any(ctx.want.values()):
            return None, None, None, None, None, None, None, None
        if ctx.fused:
            kept_dH, kept_dW = ctx.saved_tensors
            dH, dW = scale_gradients(
                kept_dH.clone() if kept_dH is not None else None,
                kept_dW.clone() if kept_dW is not None else None, dloss)
        else:
            h, W, labels, lse = ctx.saved_tensors
            dH, dW = backward(h, W, labels, lse, dloss, ctx.ignore_index,
                              ctx.chunk_rows, **ctx.variant, **ctx.want)
        return (dH, dW.to(ctx.w_dtype) if dW is not None else None, None,
                None, None, None, None, None)


class SequenceTiledMLP(torch.autograd.Function):
    """y = down(silu(gate(x)) * up(x)) over row chunks, as an autograd
    Function: forward keeps only its inputs (no L x I intermediate outlives
    a chunk); backward recomputes each chunk's gate/up activations in the
    library and returns dx (bf16) and the three weight gradients in the
    weights' dtype, computing only those autograd asks for. dy is made a
    contiguous bf16 tensor first."""

    @staticmethod
    def forward(ctx, x, Wg, Wu, Wd, chunk_rows=0):
        ctx.chunk_rows = chunk_rows
        ctx.save_for_backward(x, Wg, Wu, Wd)
        return mlp_forward(x, Wg, Wu, Wd, chunk_rows)

    @staticmethod
    def backward(ctx, dy):
        x, Wg, Wu, Wd = ctx.saved_tensors
        need = ctx.needs_input_grad
        if not any(need[:4]):
            return None, None, None, None, None
        dy = dy.to(torch.bfloat16).contiguous()
        # only the gradients autograd asks for (frozen weights: dx alone)
        dx, dWg, dWu, dWd = mlp_backward(x, Wg, Wu, Wd, dy, ctx.chunk_rows,
                                         compute_dx=need[0],
                                         compute_dWgu=need[1] or need[2],
                                         compute_dWd=need[3])
        cast = [t.to(w.dtype) if (t is not None and n) else None
                for t, w, n in ((dWg, Wg, need[1]), (dWu, Wu, need[2]),
                                (dWd, Wd, need[3]))]
        return (dx, cast[0], cast[1], cast[2], None)


def sequence_tiled_mlp(x, Wg, Wu, Wd, chunk_rows: int = 0):
    """The gated MLP down(silu(gate(x)) * up(x)) (nn.Linear weight layouts:
    Wg, Wu [I, H], Wd [H, I]; bf16) with autograd, over row chunks."""
    return SequenceTiledMLP.apply(x, Wg, Wu, Wd, chunk_rows)


def linear_cross_entropy(h, W, labels, ignore_index: int = IGNORE_INDEX,
                         chunk_rows: int = 0, fused: bool = False,
                         label_smoothing: float = 0.0, z_loss: float = 0.0):
    """Mean cross entropy of h W^T against labels (autograd). label_smoothing
    and z_loss select the loss variants of lce_forward_ex."""
    return LinearCrossEntropy.apply(h, W, labels, ignore_index, chunk_rows,
                                    fused, label_smoothing, z_loss)
