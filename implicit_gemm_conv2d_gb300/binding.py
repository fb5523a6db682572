"""Thin ctypes binding over the C ABI in include/conv.h.

Argument marshalling only: every step of the computation runs in the CUDA
library (_build/libigconv.so).  PyTorch supplies device memory and streams.
If the library is missing the functions raise; there is no fallback.

The functions named like the C entry points (conv_fwd, conv_bwd_data,
conv_bwd_filter, conv_bwd_filter_workspace_size, conv_query, ...) take
already-allocated CUDA tensors and enqueue on the current torch stream (or the
stream given).  fwd / bwd_data / bwd_filter are conveniences that allocate
the outputs (and the wgrad workspace) with torch first.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

F32, BF16 = 0, 1
ALGO_AUTO, ALGO_DIRECT, ALGO_FFMA, ALGO_TC = 0, 1, 2, 3
OP_FWD, OP_BWD_DATA, OP_BWD_FILTER, OP_BWD_BIAS, OP_FWD_WS, OP_BWD_DATA_WS, OP_BWD = 0, 1, 2, 3, 4, 5, 6
ALGO_NAMES = {0: "auto", 1: "direct", 2: "ffma", 3: "tc"}

_DT = {torch.float32: F32, torch.bfloat16: BF16}
_lock = threading.Lock()
_lib = None


class ConvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class ConvDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "IC", "OC", "H", "W", "K", "S", "relu", "dtype")]


class PlanInfo(ctypes.Structure):
    _fields_ = [("algo", ctypes.c_int32), ("launches", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("block", ctypes.c_int32), ("smem_bytes", ctypes.c_int32), ("splits", ctypes.c_int32),
                ("workspace", ctypes.c_size_t)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


EXPORTS = ["conv_fwd", "conv_bwd_data", "conv_bwd_filter_workspace_size", "conv_bwd_filter",
           "conv_status_string", "conv_out_dims", "conv_query", "conv_set_algo",
           "conv_fastdivmod_check", "conv_l2_flush", "conv_version", "conv_bwd_filter_noalloc",
           "conv_device_status", "conv_fwd_bias", "conv_bwd_bias",
           "conv_wait_selftest", "conv_query_for_device", "conv_fwd_workspace_size", "conv_fwd_ws",
           "conv_bwd_data_workspace_size", "conv_bwd_data_ws", "conv_bwd_filter_bias",
           "conv_fwd_chain2_workspace_size", "conv_fwd_chain2", "conv_query_chain2",
           "conv_bwd_chain2_workspace_size", "conv_bwd_chain2", "conv_bwd_workspace_size",
           "conv_bwd"]
STATUS_WAIT_SELFTEST = 1 << 30
NOALLOC_SCRATCH_BYTES = 16 << 20


def library_path() -> str:
    return _build.SO


def lib():
    """Load the CUDA library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built ({path} missing): run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(path)
        vp, dp, sz = ctypes.c_void_p, ctypes.POINTER(ConvDesc), ctypes.c_size_t
        L.conv_fwd.argtypes = [dp, vp, vp, vp, vp]
        L.conv_bwd_data.argtypes = [dp, vp, vp, vp, vp, vp]
        L.conv_bwd_filter_workspace_size.argtypes = [dp]
        L.conv_bwd_filter_workspace_size.restype = sz
        L.conv_bwd_filter.argtypes = [dp, vp, vp, vp, vp, vp, sz, vp]
        L.conv_status_string.argtypes = [ctypes.c_int]
        L.conv_status_string.restype = ctypes.c_char_p
        L.conv_out_dims.argtypes = [dp, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
        L.conv_query.argtypes = [ctypes.c_int, dp, ctypes.POINTER(PlanInfo)]
        L.conv_set_algo.argtypes = [ctypes.c_int, ctypes.c_int]
        L.conv_fastdivmod_check.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
        L.conv_fastdivmod_check.restype = ctypes.c_uint64
        L.conv_l2_flush.argtypes = [vp, sz, vp]
        L.conv_version.restype = ctypes.c_char_p
        L.conv_bwd_filter_noalloc.argtypes = [dp, vp, vp, vp, vp, vp]
        L.conv_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
        L.conv_fwd_bias.argtypes = [dp, vp, vp, vp, vp, vp]
        L.conv_bwd_bias.argtypes = [dp, vp, vp, vp, vp]
        L.conv_wait_selftest.argtypes = [ctypes.c_uint32, vp]
        L.conv_query_for_device.argtypes = [ctypes.c_int, dp] + [ctypes.c_int] * 4 + [ctypes.POINTER(PlanInfo)]
        L.conv_fwd_workspace_size.argtypes = [dp]
        L.conv_fwd_workspace_size.restype = sz
        L.conv_fwd_ws.argtypes = [dp, vp, vp, vp, vp, vp, sz, vp]
        L.conv_bwd_data_workspace_size.argtypes = [dp]
        L.conv_bwd_data_workspace_size.restype = sz
        L.conv_bwd_data_ws.argtypes = [dp, vp, vp, vp, vp, vp, sz, vp]
        L.conv_bwd_filter_bias.argtypes = [dp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.conv_fwd_chain2_workspace_size.argtypes = [dp, dp]
        L.conv_fwd_chain2_workspace_size.restype = sz
        L.conv_fwd_chain2.argtypes = [dp, dp] + [vp] * 8 + [sz, vp]
        L.conv_query_chain2.argtypes = [dp, dp, ctypes.POINTER(PlanInfo)]
        L.conv_bwd_chain2_workspace_size.argtypes = [dp, dp]
        L.conv_bwd_chain2_workspace_size.restype = sz
        L.conv_bwd_chain2.argtypes = [dp, dp] + [vp] * 11 + [vp, sz, vp]
        L.conv_bwd_workspace_size.argtypes = [dp]
        L.conv_bwd_workspace_size.restype = sz
        L.conv_bwd.argtypes = [dp] + [vp] * 8 + [sz, vp]
        _lib = L
        return L


def status_string(status: int) -> str:
    return lib().conv_status_string(int(status)).decode()


def _check(rc: int, where: str):
    if rc != 0:
        raise ConvError(rc, where)


def make_desc(B, IC, OC, H, W, K, S, relu, dtype) -> ConvDesc:
    if isinstance(dtype, torch.dtype):
        dtype = _DT[dtype]
    return ConvDesc(int(B), int(IC), int(OC), int(H), int(W), int(K), int(S), int(bool(relu)), int(dtype))


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def out_dims(desc: ConvDesc):
    oh, ow = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().conv_out_dims(ctypes.byref(desc), ctypes.byref(oh), ctypes.byref(ow)), "conv_out_dims")
    return oh.value, ow.value


def conv_fwd(desc: ConvDesc, x, w, y, stream=None) -> None:
    _check(lib().conv_fwd(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(y), _stream(stream)), "conv_fwd")


def conv_fwd_bias(desc: ConvDesc, x, w, bias, y, stream=None) -> None:
    _check(lib().conv_fwd_bias(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(bias), _ptr(y), _stream(stream)),
           "conv_fwd_bias")


def conv_bwd_bias(desc: ConvDesc, dy, y, db, stream=None) -> None:
    _check(lib().conv_bwd_bias(ctypes.byref(desc), _ptr(dy), _ptr(y), _ptr(db), _stream(stream)),
           "conv_bwd_bias")


def conv_bwd_data(desc: ConvDesc, dy, w, y, dx, stream=None) -> None:
    _check(lib().conv_bwd_data(ctypes.byref(desc), _ptr(dy), _ptr(w), _ptr(y), _ptr(dx), _stream(stream)),
           "conv_bwd_data")


def conv_fwd_workspace_size(desc: ConvDesc) -> int:
    return int(lib().conv_fwd_workspace_size(ctypes.byref(desc)))


def conv_fwd_ws(desc: ConvDesc, x, w, bias, y, workspace, stream=None) -> None:
    """The forward with a caller-provided workspace (bias may be None)."""
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().conv_fwd_ws(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(bias), _ptr(y), _ptr(workspace), nbytes,
                             _stream(stream)), "conv_fwd_ws")


def conv_bwd_data_workspace_size(desc: ConvDesc) -> int:
    return int(lib().conv_bwd_data_workspace_size(ctypes.byref(desc)))


def conv_bwd_data_ws(desc: ConvDesc, dy, w, y, dx, workspace, stream=None) -> None:
    """d_input with a caller-provided workspace."""
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().conv_bwd_data_ws(ctypes.byref(desc), _ptr(dy), _ptr(w), _ptr(y), _ptr(dx), _ptr(workspace),
                                  nbytes, _stream(stream)), "conv_bwd_data_ws")


def conv_bwd_filter_workspace_size(desc: ConvDesc) -> int:
    return int(lib().conv_bwd_filter_workspace_size(ctypes.byref(desc)))


def conv_bwd_filter(desc: ConvDesc, x, dy, y, dw, workspace, stream=None) -> None:
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().conv_bwd_filter(ctypes.byref(desc), _ptr(x), _ptr(dy), _ptr(y), _ptr(dw),
                                 _ptr(workspace), nbytes, _stream(stream)), "conv_bwd_filter")


def conv_bwd_filter_bias(desc: ConvDesc, x, dy, y, dw, db, workspace, stream=None) -> None:
    """Weight and bias gradients in one pass over g (the same workspace as conv_bwd_filter)."""
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().conv_bwd_filter_bias(ctypes.byref(desc), _ptr(x), _ptr(dy), _ptr(y), _ptr(dw), _ptr(db),
                                      _ptr(workspace), nbytes, _stream(stream)), "conv_bwd_filter_bias")


def conv_fwd_chain2_workspace_size(d1: ConvDesc, d2: ConvDesc) -> int:
    return int(lib().conv_fwd_chain2_workspace_size(ctypes.byref(d1), ctypes.byref(d2)))


def conv_fwd_chain2(d1: ConvDesc, d2: ConvDesc, x, w1, bias1, w2, bias2, y1, y2, workspace, stream=None) -> None:
    """Two-layer forward chain (layer 2's input is layer 1's output); biases may be None."""
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().conv_fwd_chain2(ctypes.byref(d1), ctypes.byref(d2), _ptr(x), _ptr(w1), _ptr(bias1), _ptr(w2),
                                 _ptr(bias2), _ptr(y1), _ptr(y2), _ptr(workspace), nbytes, _stream(stream)),
           "conv_fwd_chain2")


def conv_bwd_chain2_workspace_size(d1: ConvDesc, d2: ConvDesc) -> int:
    return int(lib().conv_bwd_chain2_workspace_size(ctypes.byref(d1), ctypes.byref(d2)))


def conv_bwd_chain2(d1: ConvDesc, d2: ConvDesc, x1, w1, y1, w2, y2, dy2, dx1, dw1, db1, dw2, db2, workspace,
                    stream=None) -> None:
    """Backward of the two-layer stack (dx1, db1, db2 may be None: not computed)."""
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().conv_bwd_chain2(ctypes.byref(d1), ctypes.byref(d2), _ptr(x1), _ptr(w1), _ptr(y1), _ptr(w2),
                                 _ptr(y2), _ptr(dy2), _ptr(dx1), _ptr(dw1), _ptr(db1), _ptr(dw2), _ptr(db2),
                                 _ptr(workspace), nbytes, _stream(stream)),
           "conv_bwd_chain2")


def conv_query_chain2(d1: ConvDesc, d2: ConvDesc) -> dict:
    info = PlanInfo()
    _check(lib().conv_query_chain2(ctypes.byref(d1), ctypes.byref(d2), ctypes.byref(info)), "conv_query_chain2")
    d = info.as_dict()
    d["algo_name"] = ALGO_NAMES.get(d["algo"], "?")
    return d


def conv_bwd_workspace_size(desc: ConvDesc) -> int:
    return int(lib().conv_bwd_workspace_size(ctypes.byref(desc)))


def conv_bwd(desc: ConvDesc, x, dy, w, y, dx, dw, db, workspace, stream=None) -> None:
    """The whole backward: dx, dw and (db not None) db, d_input and wgrad in one launch."""
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().conv_bwd(ctypes.byref(desc), _ptr(x), _ptr(dy), _ptr(w), _ptr(y), _ptr(dx), _ptr(dw), _ptr(db),
                          _ptr(workspace), nbytes, _stream(stream)), "conv_bwd")


def conv_bwd_filter_noalloc(desc: ConvDesc, x, dy, y, dw, stream=None) -> None:
    """Weight gradient with no workspace argument and no allocation: the split-K
    partials use the library's fixed scratch array (see include/conv.h).  For
    callers that cannot allocate device memory; concurrent calls race."""
    _check(lib().conv_bwd_filter_noalloc(ctypes.byref(desc), _ptr(x), _ptr(dy), _ptr(y), _ptr(dw),
                                         _stream(stream)), "conv_bwd_filter_noalloc")


def conv_query(op: int, desc: ConvDesc) -> dict:
    info = PlanInfo()
    _check(lib().conv_query(int(op), ctypes.byref(desc), ctypes.byref(info)), "conv_query")
    d = info.as_dict()
    d["algo_name"] = ALGO_NAMES.get(d["algo"], "?")
    return d


GB300 = dict(sms=152, smem_optin=232448, cc_major=10, cc_minor=3)


def conv_query_for_device(op: int, desc: ConvDesc, sms: int, smem_optin: int, cc_major: int,
                          cc_minor: int) -> dict:
    """The plan for a device described by its properties (host only, no CUDA call)."""
    info = PlanInfo()
    _check(lib().conv_query_for_device(int(op), ctypes.byref(desc), int(sms), int(smem_optin), int(cc_major),
                                       int(cc_minor), ctypes.byref(info)), "conv_query_for_device")
    d = info.as_dict()
    d["algo_name"] = ALGO_NAMES.get(d["algo"], "?")
    return d


def conv_set_algo(op: int, algo: int) -> None:
    _check(lib().conv_set_algo(int(op), int(algo)), "conv_set_algo")


def conv_fastdivmod_check(d: int, lo: int, hi: int) -> int:
    return int(lib().conv_fastdivmod_check(d, lo, hi))


def conv_l2_flush(buf, stream=None) -> None:
    _check(lib().conv_l2_flush(_ptr(buf), buf.numel() * buf.element_size(), _stream(stream)),
           "conv_l2_flush")


def conv_device_status(reset: bool = False) -> int:
    """Timeout bits set by the tensor-core kernels (0 = none).  Synchronises."""
    v = ctypes.c_uint32()
    _check(lib().conv_device_status(ctypes.byref(v), int(reset)), "conv_device_status")
    return v.value


def conv_wait_selftest(max_sleeps: int, stream=None) -> None:
    """Run the bounded-wait self-test kernel (see include/conv.h); its timeout sets
    STATUS_WAIT_SELFTEST in conv_device_status()."""
    _check(lib().conv_wait_selftest(int(max_sleeps), _stream(stream)), "conv_wait_selftest")


def conv_version() -> str:
    return lib().conv_version().decode()


# ---- allocating conveniences -----------------------------------------------------------
def _desc_from(x_shape, w_shape, S, relu, dtype):
    B, IC, H, W = x_shape
    OC, IC2, K, K2 = w_shape
    if IC2 != IC or K2 != K:
        raise ValueError("x / w shapes disagree")
    return make_desc(B, IC, OC, H, W, K, S, relu, dtype)


def fwd(x, w, S: int, relu: bool, stream=None, bias=None):
    desc = _desc_from(x.shape, w.shape, S, relu, x.dtype)
    oh, ow = out_dims(desc)
    y = torch.empty((x.shape[0], w.shape[0], oh, ow), dtype=x.dtype, device=x.device)
    if bias is None:
        conv_fwd(desc, x, w, y, stream)
    else:
        conv_fwd_bias(desc, x, w, bias, y, stream)
    return y


def bias_desc(dy_shape, relu: bool, dtype) -> ConvDesc:
    """A descriptor for the bias gradient of an output of shape (B, OC, OH, OW): the
    reduction needs only those sizes, so a 1x1, stride-1 window over an OH x OW input
    stands for the layer."""
    B, OC, OH, OW = dy_shape
    return make_desc(B, 1, OC, OH, OW, 1, 1, relu, dtype)


def bwd_bias(dy, y, relu: bool, stream=None):
    db = torch.empty((dy.shape[1],), dtype=dy.dtype, device=dy.device)
    conv_bwd_bias(bias_desc(dy.shape, relu, dy.dtype), dy, y if relu else None, db, stream)
    return db


def bwd_data(dy, w, y, H: int, W: int, S: int, relu: bool, stream=None):
    B, OC = dy.shape[:2]
    OC2, IC, K, _ = w.shape
    desc = make_desc(B, IC, OC, H, W, K, S, relu, dy.dtype)
    dx = torch.empty((B, IC, H, W), dtype=dy.dtype, device=dy.device)
    conv_bwd_data(desc, dy, w, y if relu else None, dx, stream)
    return dx


def bwd_filter(x, dy, y, K: int, S: int, relu: bool, stream=None, workspace=None):
    B, IC, H, W = x.shape
    OC = dy.shape[1]
    desc = make_desc(B, IC, OC, H, W, K, S, relu, x.dtype)
    dw = torch.empty((OC, IC, K, K), dtype=x.dtype, device=x.device)
    need = conv_bwd_filter_workspace_size(desc)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    conv_bwd_filter(desc, x, dy, y if relu else None, dw, workspace, stream)
    return dw
