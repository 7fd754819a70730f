"""Float64 CPU oracle for the chunked LM-head cross-entropy.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product path
(``chunked_lm_head_gemm_gb300``) does not import it and shares no code with
it. The arithmetic lives in ``lce_oracle.c`` (plain C, float64, pthreads);
this module only compiles it with gcc and marshals arguments.

What it follows: "Training Beyond 1M Tokens" (TRL guide), sections "The loss
is the first thing to break" (logits = hidden x LM-head weights, then a
cross entropy against the labels) and "The massive logits matrix: chunk it"
(the loss is a sum over rows; the softmax runs along one row's vocabulary).
The reduction the pages leave open is: mean over rows whose label is neither
ignore_index nor outside [0, V); 0 when no row is valid.

Loss variants (not on the pages, which define only the plain cross entropy;
both 0 by default): ``label_smoothing`` eps takes the cross entropy against
the target (1 - eps) onehot + eps / V, and ``z_loss`` adds z_loss * lse^2
to each valid row's loss.

Parity of every function here is pinned in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lce_oracle.c")
_SOURCES = [_SRC, os.path.join(_HERE, "mlp_oracle.c")]
_LIB_PATH = os.path.join(_HERE, "liblce_oracle.so")
_lib = None
_lock = threading.Lock()

# Status codes returned by the C functions.
OK = 0
BAD_ARG = 1
LABEL_RANGE = 4
NO_MEMORY = 7

DT_BF16, DT_F32, DT_F64 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle's C sources into liblce_oracle.so (gcc, -O2)."""
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(f)
                    for f in _SOURCES)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-fPIC", "-shared",
                    "-pthread", "-o", tmp, *_SOURCES, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Open a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    p, i64, i32, f64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                        ctypes.c_double)
    lib.lce_oracle_forward.argtypes = [p, p, i32, p, i64, i64, i64, i64,
                                       f64, f64, i32, p, p, p, p]
    lib.lce_oracle_forward.restype = i32
    lib.lce_oracle_backward.argtypes = [p, p, i32, p, i64, i64, i64, i64,
                                        f64, f64, f64, i32, p, p, p, i64]
    lib.lce_oracle_backward.restype = i32
    lib.lce_oracle_rows.argtypes = [p, p, i32, p, i64, i64, i64, i64, f64,
                                    f64, f64, p, i64, i32, p, p, p]
    lib.lce_oracle_rows.restype = i32
    lib.lce_oracle_forward_backward.argtypes = [p, p, i32, p, i64, i64, i64,
                                                i64, f64, f64, f64, i32, p, p,
                                                p, p, p, p, p, i64]
    lib.lce_oracle_forward_backward.restype = i32
    lib.lce_oracle_count_valid.argtypes = [p, i64, i64, i64, p]
    lib.lce_oracle_count_valid.restype = i64
    if hasattr(lib, "mlp_oracle"):
        lib.mlp_oracle.argtypes = [p, p, p, p, i32, i64, i64, i64, p, i32, p,
                                   p, p, p, p]
        lib.mlp_oracle.restype = i32
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _as_input(x):
    """Return (contiguous numpy array, dtype code) for h or W.

    Accepts numpy float32/float64 arrays and torch CPU tensors of dtype
    bfloat16/float32/float64 (bf16 is passed as its raw 16-bit patterns)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), DT_BF16
            x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, DT_F32
    if x.dtype == np.float64:
        return x, DT_F64
    if x.dtype == np.uint16:
        return x, DT_BF16
    raise TypeError(f"oracle input dtype {x.dtype} not supported")


def _labels(y):
    try:
        import torch
        if isinstance(y, torch.Tensor):
            y = y.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(y, dtype=np.int64)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def forward(h, W, labels, ignore_index: int = -100, nthreads: int | None = None,
            label_smoothing: float = 0.0, z_loss: float = 0.0):
    """Returns dict(loss, lse[L], zy[L], n_valid, status) in float64."""
    hn, dt = _as_input(h)
    Wn, dt2 = _as_input(W)
    if dt != dt2:
        raise TypeError("h and W must have the same dtype")
    y = _labels(labels)
    L, H = hn.shape
    V = Wn.shape[0]
    assert Wn.shape[1] == H and y.shape == (L,)
    lse = np.empty(L, np.float64)
    zy = np.empty(L, np.float64)
    loss = np.zeros(1, np.float64)
    nv = np.zeros(1, np.int64)
    st = _load().lce_oracle_forward(_ptr(hn), _ptr(Wn), dt, _ptr(y), L, H, V,
                                    ignore_index, float(label_smoothing),
                                    float(z_loss),
                                    nthreads or default_threads(),
                                    _ptr(lse), _ptr(zy), _ptr(loss), _ptr(nv))
    if st not in (OK, LABEL_RANGE):
        raise RuntimeError(f"lce_oracle_forward status {st}")
    return dict(loss=float(loss[0]), lse=lse, zy=zy, n_valid=int(nv[0]),
                status=st)


def backward(h, W, labels, dloss: float = 1.0, ignore_index: int = -100,
             want_dH: bool = True, want_dW: bool = True, vrows=None,
             nthreads: int | None = None, label_smoothing: float = 0.0,
             z_loss: float = 0.0):
    """Returns dict(dH[L,H] or None, dW or None, status) in float64.

    dW is [V,H], or [len(vrows), H] holding rows dW[vrows] when vrows is
    given."""
    hn, dt = _as_input(h)
    Wn, dt2 = _as_input(W)
    if dt != dt2:
        raise TypeError("h and W must have the same dtype")
    y = _labels(labels)
    L, H = hn.shape
    V = Wn.shape[0]
    vr = None if vrows is None else np.ascontiguousarray(vrows, dtype=np.int64)
    dH = np.empty((L, H), np.float64) if want_dH else None
    nvr = V if vr is None else vr.shape[0]
    dW = np.empty((nvr, H), np.float64) if want_dW else None
    st = _load().lce_oracle_backward(_ptr(hn), _ptr(Wn), dt, _ptr(y), L, H, V,
                                     ignore_index, float(label_smoothing),
                                     float(z_loss), float(dloss),
                                     nthreads or default_threads(), _ptr(dH),
                                     _ptr(dW), _ptr(vr),
                                     0 if vr is None else nvr)
    if st not in (OK, LABEL_RANGE):
        raise RuntimeError(f"lce_oracle_backward status {st}")
    return dict(dH=dH, dW=dW, status=st)


def rows(h, W, labels, rows, dloss: float = 1.0, ignore_index: int = -100,
         want_dH: bool = True, nthreads: int | None = None,
         label_smoothing: float = 0.0, z_loss: float = 0.0):
    """Selected rows of a problem of any size (N counted over all labels).

    Returns dict(lse[n], zy[n], dH[n,H] or None, status) in float64."""
    hn, dt = _as_input(h)
    Wn, dt2 = _as_input(W)
    if dt != dt2:
        raise TypeError("h and W must have the same dtype")
    y = _labels(labels)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    L, H = hn.shape
    V = Wn.shape[0]
    n = r.shape[0]
    lse = np.empty(n, np.float64)
    zy = np.empty(n, np.float64)
    dH = np.empty((n, H), np.float64) if want_dH else None
    st = _load().lce_oracle_rows(_ptr(hn), _ptr(Wn), dt, _ptr(y), L, H, V,
                                 ignore_index, float(label_smoothing),
                                 float(z_loss), float(dloss), _ptr(r), n,
                                 nthreads or default_threads(), _ptr(lse),
                                 _ptr(zy), _ptr(dH))
    if st not in (OK, LABEL_RANGE):
        raise RuntimeError(f"lce_oracle_rows status {st}")
    return dict(lse=lse, zy=zy, dH=dH, status=st)


def forward_backward(h, W, labels, dloss: float = 1.0,
                     ignore_index: int = -100, want_dH: bool = True,
                     want_dW: bool = True, vrows=None,
                     nthreads: int | None = None,
                     label_smoothing: float = 0.0, z_loss: float = 0.0):
    """forward() and backward() of the same problem from one pass over the
    logits. Returns dict(loss, lse, zy, n_valid, dH, dW, status)."""
    hn, dt = _as_input(h)
    Wn, dt2 = _as_input(W)
    if dt != dt2:
        raise TypeError("h and W must have the same dtype")
    y = _labels(labels)
    L, H = hn.shape
    V = Wn.shape[0]
    assert Wn.shape[1] == H and y.shape == (L,)
    vr = None if vrows is None else np.ascontiguousarray(vrows, dtype=np.int64)
    lse = np.empty(L, np.float64)
    zy = np.empty(L, np.float64)
    loss = np.zeros(1, np.float64)
    nv = np.zeros(1, np.int64)
    dH = np.empty((L, H), np.float64) if want_dH else None
    nvr = V if vr is None else vr.shape[0]
    dW = np.empty((nvr, H), np.float64) if want_dW else None
    st = _load().lce_oracle_forward_backward(
        _ptr(hn), _ptr(Wn), dt, _ptr(y), L, H, V, ignore_index,
        float(label_smoothing), float(z_loss), float(dloss),
        nthreads or default_threads(), _ptr(lse), _ptr(zy), _ptr(loss),
        _ptr(nv), _ptr(dH), _ptr(dW), _ptr(vr), 0 if vr is None else nvr)
    if st not in (OK, LABEL_RANGE):
        raise RuntimeError(f"lce_oracle_forward_backward status {st}")
    return dict(loss=float(loss[0]), lse=lse, zy=zy, n_valid=int(nv[0]),
                dH=dH, dW=dW, status=st)


def count_valid(labels, V: int, ignore_index: int = -100):
    """Returns (N, any_label_out_of_range)."""
    y = _labels(labels)
    bad = ctypes.c_int(0)
    n = _load().lce_oracle_count_valid(_ptr(y), y.shape[0], V, ignore_index,
                                       ctypes.byref(bad))
    return int(n), bool(bad.value)


def mlp(x, Wg, Wu, Wd, dy=None, want_dx: bool = True, want_dW: bool = True,
        nthreads: int | None = None):
    """Gated MLP y = (silu(x Wg^T) * (x Wu^T)) Wd^T in float64, and its
    backward for dy (float64-widened) when given.

    x [L,H]; Wg, Wu [I,H]; Wd [H,I] (one dtype). Returns dict(y, dx, dWg,
    dWu, dWd); gradients are None without dy or when not wanted."""
    xn, dt = _as_input(x)
    arrs = [_as_input(w) for w in (Wg, Wu, Wd)]
    if any(a[1] != dt for a in arrs):
        raise TypeError("x and the weights must have the same dtype")
    gn, un, dn = (a[0] for a in arrs)
    L, H = xn.shape
    I = gn.shape[0]
    assert gn.shape == (I, H) and un.shape == (I, H) and dn.shape == (H, I)
    y = np.empty((L, H), np.float64)
    dyn = None
    dx = dWg = dWu = dWd = None
    if dy is not None:
        try:
            import torch
            if isinstance(dy, torch.Tensor):
                dy = dy.detach().cpu().double().numpy()
        except ImportError:  # pragma: no cover
            pass
        dyn = np.ascontiguousarray(dy, dtype=np.float64)
        assert dyn.shape == (L, H)
        if want_dx:
            dx = np.empty((L, H), np.float64)
        if want_dW:
            dWg = np.empty((I, H), np.float64)
            dWu = np.empty((I, H), np.float64)
            dWd = np.empty((H, I), np.float64)
    st = _load().mlp_oracle(_ptr(xn), _ptr(gn), _ptr(un), _ptr(dn), dt, L, H,
                            I, _ptr(dyn), nthreads or default_threads(),
                            _ptr(y), _ptr(dx), _ptr(dWg), _ptr(dWu),
                            _ptr(dWd))
    if st != OK:
        raise RuntimeError(f"mlp_oracle status {st}")
    return dict(y=y, dx=dx, dWg=dWg, dWu=dWu, dWd=dWd)
