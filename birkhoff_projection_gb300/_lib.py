"""ctypes loader for libbirkhoff4.so (the C ABI of include/birkhoff4.h).

Only argument marshalling lives here.  If the library cannot be built or
loaded, every call raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

_lock = threading.Lock()
_lib = None

B4_OK, B4_EINVAL, B4_ECUDA, B4_ENOTIMPL, B4_ESCRATCH = 0, 1, 2, 3, 4
B4_F32, B4_BF16 = 0, 1
B4_SCHED_DEFAULT, B4_SCHED_QUEUE, B4_SCHED_LANE, B4_SCHED_LANES4 = 0, 1, 2, 3

# Every function the header declares, with its ctypes signature.
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
SIGNATURES = {
    "birkhoff4_forward": (_int, [_vp, _vp, _vp, _i64, _vp]),
    "birkhoff4_forward_bf16": (_int, [_vp, _vp, _vp, _i64, _vp]),
    "birkhoff4_forward_ex": (_int, [_vp, _vp, _vp, _i64, _vp, _vp]),
    "birkhoff4_backward": (_int, [_vp, _vp, _vp, _vp, _i64, _vp]),
    "birkhoff4_backward_bf16": (_int, [_vp, _vp, _vp, _vp, _i64, _vp]),
    "birkhoff4_forward_backward": (_int, [_vp, _vp, _vp, _vp, _i64, _vp]),
    "birkhoff4_forward_backward_bf16": (_int, [_vp, _vp, _vp, _vp, _i64, _vp]),
    "birkhoff4_forward_backward_ex": (_int, [_vp, _vp, _vp, _vp, _i64, _vp, _vp]),
    "birkhoff4_forward_backward_host": (_int, [_vp, _vp, _vp, _vp, _i64, ctypes.c_int32, _vp,
                                               ctypes.c_size_t, _vp, ctypes.c_int32]),
    "birkhoff4_forward_backward_host_static": (_int, [_vp, _vp, _vp, _vp, _i64, ctypes.c_int32,
                                                      _i64, _vp, ctypes.c_int32]),
    "birkhoff4_forward_nxn": (_int, [_vp, _vp, _vp, ctypes.c_int32, _i64, _vp]),
    "birkhoff4_forward_backward_mapped": (_int, [_vp, _vp, _vp, _vp, _i64, ctypes.c_int32, _vp]),
    "eot_workspace_bytes": (ctypes.c_size_t, [_i64, _i64, ctypes.c_int32, ctypes.c_int32]),
    "eot_update": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_int32, ctypes.c_float,
                          ctypes.c_int32, _vp, ctypes.c_size_t, _vp]),
    "eot_transport_workspace_bytes": (ctypes.c_size_t, [_i64, _i64, ctypes.c_int32]),
    "eot_transport": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                             ctypes.c_int32, ctypes.c_float, _vp, ctypes.c_size_t, _vp]),
    "eot_apply_plan_workspace_bytes": (ctypes.c_size_t, [_i64, _i64, ctypes.c_int32, ctypes.c_int32]),
    "eot_apply_plan": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int32, _vp, _vp, _i64,
                              _i64, ctypes.c_int32, ctypes.c_float, _vp, ctypes.c_size_t, _vp]),
    "eot_transport_schedule": (_int, [_i64, ctypes.c_int32, ctypes.c_int32, _vp]),
    "eot_hvp_workspace_bytes": (ctypes.c_size_t, [_i64, _i64, ctypes.c_int32]),
    "eot_hvp": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_int32,
                       ctypes.c_float, ctypes.c_int32, _vp, ctypes.c_size_t, _vp]),
    "eot_sinkhorn": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_int32,
                            ctypes.c_float, ctypes.c_int32, ctypes.c_int32, _vp, ctypes.c_size_t,
                            _vp]),
    "birkhoff4_backward_nxn": (_int, [_vp, _vp, _vp, ctypes.c_int32, _i64, _vp]),
    "birkhoff4_sinkhorn": (_int, [_vp, _vp, _int, _i64, _vp]),
    "birkhoff4_sinkhorn_bf16": (_int, [_vp, _vp, _int, _i64, _vp]),
    "birkhoff4_strerror": (ctypes.c_char_p, [_int]),
    "birkhoff4_version": (_int, []),
    "birkhoff4_last_cuda_error": (_int, []),
    "birkhoff4_device_status": (_int, [ctypes.POINTER(ctypes.c_uint), _int]),
    "birkhoff4_selftest_wait_timeout": (_int, [_i64]),
    "birkhoff4_mufu_probe": (_int, [ctypes.POINTER(ctypes.c_float), _int, _int, _vp]),
}


class Opts(ctypes.Structure):
    """birkhoff4_opts."""
    _fields_ = [
        ("in_dtype", ctypes.c_int32),
        ("out_dtype", ctypes.c_int32),
        ("max_evals", ctypes.c_int32),
        ("tol", ctypes.c_float),
        ("evals_out", ctypes.c_void_p),
        ("nonconv_count", ctypes.c_void_p),
        ("schedule", ctypes.c_int32),
    ]


class Birkhoff4Error(RuntimeError):
    pass


def lib():
    """The loaded library (built with nvcc on first use if missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build()
        if not os.path.exists(path):
            raise Birkhoff4Error("libbirkhoff4.so was not built")
        handle = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
        return handle


def library_path() -> str:
    return _build.LIB_PATH


def check(status: int, what: str) -> None:
    if status != B4_OK:
        L = lib()
        msg = L.birkhoff4_strerror(status).decode()
        if status == B4_ECUDA:
            msg += " (cudaError %d)" % L.birkhoff4_last_cuda_error()
        raise Birkhoff4Error("%s: %s" % (what, msg))
