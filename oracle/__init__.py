"""fp64 CPU oracle for the conv2d layer (forward + bias + ReLU, d_input, wgrad,
bias grad).

TEST INFRASTRUCTURE ONLY.  The product path never imports this package; only
the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg do.

The arithmetic lives in ``conv_ref.c`` (plain C, direct loops, fp64); this
module builds it with gcc on first use and marshals numpy arrays in and out.
Definitions follow PufferLib PR #522 ("Speedups to gemm_conv_forward and
gemm_conv_backward kernels"), whose layer-1 and layer-2 bench blocks name the
forward, "backward wgrad" and "backward d_input" results and print the shapes
11x15 K=5 S=3 -> 3x4 (relu=1) and 3x4 K=3 S=1 -> 1x2 (relu=0); the bias is the
per-output-channel conv bias whose gradient the same PR's "n3_conv_bias_grad"
blocks time (added before the activation in the forward; its gradient is the
sum of the masked output gradient over batch and positions).

Every function returns ``(out, den)`` where ``den`` holds, per output element,
the sum of |term| over the products that element sums; the normalised error of
a result is ``|out - ref| / den``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv_ref.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


class _Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("IC", ctypes.c_int64), ("OC", ctypes.c_int64),
                ("H", ctypes.c_int64), ("W", ctypes.c_int64), ("K", ctypes.c_int64),
                ("S", ctypes.c_int64), ("relu", ctypes.c_int32)]


def build(force: bool = False) -> str:
    """Compile conv_ref.c into _build/liboracle.so (gcc, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def bind(path: str):
    """Load a build of conv_ref.c from ``path``; pass the result as ``lib=`` to
    run the same wrappers against it (used by the planted-mistake tests)."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    sp = ctypes.POINTER(_Shape)
    lib.oracle_conv_fwd.argtypes = [sp, dp, dp, dp, dp, ctypes.c_int]
    lib.oracle_conv_bwd_data.argtypes = [sp, dp, dp, dp, dp, dp, ctypes.c_int]
    lib.oracle_conv_bwd_filter.argtypes = [sp, dp, dp, dp, dp, dp, ctypes.c_int]
    lib.oracle_conv_fwd_bias.argtypes = [sp, dp, dp, dp, dp, dp, ctypes.c_int]
    lib.oracle_conv_bwd_bias.argtypes = [sp, dp, dp, dp, dp, ctypes.c_int]
    for f in (lib.oracle_conv_fwd, lib.oracle_conv_bwd_data, lib.oracle_conv_bwd_filter,
              lib.oracle_conv_fwd_bias, lib.oracle_conv_bwd_bias):
        f.restype = ctypes.c_int
    lib.oracle_out_dim.argtypes = [ctypes.c_int64] * 3
    lib.oracle_out_dim.restype = ctypes.c_int64
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def out_dim(n: int, K: int, S: int) -> int:
    """Spatial output size of one axis (no padding)."""
    return int(_load().oracle_out_dim(n, K, S))


def _shape(B, IC, OC, H, W, K, S, relu):
    return _Shape(B, IC, OC, H, W, K, S, 1 if relu else 0)


def conv_fwd(x, w, S: int, relu: bool, nthreads: int | None = None, lib=None, bias=None):
    """y = act(conv(x, w) + bias) with x (B,IC,H,W), w (OC,IC,K,K), bias (OC,) or None
    (no bias term).  Returns (y, den); den includes |bias[oc]|."""
    x, w = _f64(x), _f64(w)
    B, IC, H, W = x.shape
    OC, IC2, K, K2 = w.shape
    assert IC2 == IC and K2 == K
    OH, OW = out_dim(H, K, S), out_dim(W, K, S)
    y = np.empty((B, OC, OH, OW))
    den = np.empty_like(y)
    lib = lib or _load()
    shape = ctypes.byref(_shape(B, IC, OC, H, W, K, S, relu))
    if bias is None:
        rc = lib.oracle_conv_fwd(shape, _ptr(x), _ptr(w), _ptr(y), _ptr(den),
                                 nthreads or default_threads())
    else:
        bias = _f64(bias)
        assert bias.shape == (OC,)
        rc = lib.oracle_conv_fwd_bias(shape, _ptr(x), _ptr(w), _ptr(bias), _ptr(y), _ptr(den),
                                      nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_conv_fwd rejected the arguments (rc={rc})")
    return y, den


def conv_bwd_data(dy, w, y, H: int, W: int, S: int, relu: bool, nthreads: int | None = None,
                  lib=None):
    """dx (B,IC,H,W) from dy (B,OC,OH,OW); y masks dy when relu.  Returns (dx, den)."""
    dy, w = _f64(dy), _f64(w)
    y = _f64(y) if (relu and y is not None) else None
    B, OC, OH, OW = dy.shape
    OC2, IC, K, _ = w.shape
    assert OC2 == OC and out_dim(H, K, S) == OH and out_dim(W, K, S) == OW
    dx = np.empty((B, IC, H, W))
    den = np.empty_like(dx)
    rc = (lib or _load()).oracle_conv_bwd_data(ctypes.byref(_shape(B, IC, OC, H, W, K, S, relu)),
                                      _ptr(dy), _ptr(w), _ptr(y), _ptr(dx), _ptr(den),
                                      nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_conv_bwd_data rejected the arguments (rc={rc})")
    return dx, den


def conv_bwd_filter(x, dy, y, K: int, S: int, relu: bool, nthreads: int | None = None,
                    lib=None):
    """dw (OC,IC,K,K) from x and dy; y masks dy when relu.  Returns (dw, den)."""
    x, dy = _f64(x), _f64(dy)
    y = _f64(y) if (relu and y is not None) else None
    B, IC, H, W = x.shape
    B2, OC, OH, OW = dy.shape
    assert B2 == B and out_dim(H, K, S) == OH and out_dim(W, K, S) == OW
    dw = np.empty((OC, IC, K, K))
    den = np.empty_like(dw)
    rc = (lib or _load()).oracle_conv_bwd_filter(ctypes.byref(_shape(B, IC, OC, H, W, K, S, relu)),
                                        _ptr(x), _ptr(dy), _ptr(y), _ptr(dw), _ptr(den),
                                        nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_conv_bwd_filter rejected the arguments (rc={rc})")
    return dw, den


def conv_bwd_bias(dy, y, relu: bool, nthreads: int | None = None, lib=None):
    """db (OC,) = sum over b, oh, ow of dy (B,OC,OH,OW), masked by y > 0 when relu.
    Returns (db, den)."""
    dy = _f64(dy)
    y = _f64(y) if (relu and y is not None) else None
    B, OC, OH, OW = dy.shape
    db = np.empty((OC,))
    den = np.empty_like(db)
    # The shape record wants a window; K = S = 1 over an OH x OW input reproduces OH x OW.
    rc = (lib or _load()).oracle_conv_bwd_bias(ctypes.byref(_shape(B, 1, OC, OH, OW, 1, 1, relu)),
                                      _ptr(dy), _ptr(y), _ptr(db), _ptr(den),
                                      nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_conv_bwd_bias rejected the arguments (rc={rc})")
    return db, den


def normalised_error(out, ref, den) -> float:
    """max over elements of |out - ref| / den; where den == 0, out must equal ref exactly
    (any mismatch there counts as infinite error)."""
    out = np.asarray(out, dtype=np.float64)
    diff = np.abs(out - ref)
    zero = den == 0
    if np.any(diff[zero] != 0):
        return float("inf")
    if not np.any(~zero):
        return 0.0
    return float(np.max(diff[~zero] / den[~zero]))
