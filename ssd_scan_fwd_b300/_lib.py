"""ctypes view of the C ABI declared in include/ssd.h.

Argument marshalling only: this module loads ``libssd_scan_fwd.so`` (built
in-tree by ``ssd_scan_fwd_b300.build``) and mirrors its struct and entry
points.  It raises if the library is missing -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssd_scan_fwd.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "ssd.h")

SSD_OK = 0
SSD_ERR_INVALID_ARG = 1
SSD_ERR_UNSUPPORTED = 2
SSD_ERR_WORKSPACE = 3
SSD_ERR_CUDA = 4
SSD_ERR_TIMEOUT = 5

SSD_DTYPE_F32 = 0
SSD_DTYPE_BF16 = 1

SSD_ALGO_AUTO = 0
SSD_ALGO_CHUNKED = 1
SSD_ALGO_FUSED = 2

ALGOS = {"auto": SSD_ALGO_AUTO, "chunked": SSD_ALGO_CHUNKED, "fused": SSD_ALGO_FUSED}


class SsdFwdArgs(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int64),
        ("seqlen", ctypes.c_int64),
        ("nheads", ctypes.c_int64),
        ("headdim", ctypes.c_int64),
        ("ngroups", ctypes.c_int64),
        ("dstate", ctypes.c_int64),
        ("io_dtype", ctypes.c_int32),
        ("algo", ctypes.c_int32),
        ("chunk_size", ctypes.c_int64),
        ("x", ctypes.c_void_p),
        ("dt", ctypes.c_void_p),
        ("A", ctypes.c_void_p),
        ("Bm", ctypes.c_void_p),
        ("Cm", ctypes.c_void_p),
        ("D", ctypes.c_void_p),
        ("init_state", ctypes.c_void_p),
        ("y", ctypes.c_void_p),
        ("final_state", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
    ]


class SsdFwdExArgs(ctypes.Structure):
    _fields_ = [
        ("base", SsdFwdArgs),
        ("dt_bias", ctypes.c_void_p),
        ("dt_softplus", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("z", ctypes.c_void_p),
    ]


class SsdStepArgs(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int64),
        ("nheads", ctypes.c_int64),
        ("headdim", ctypes.c_int64),
        ("ngroups", ctypes.c_int64),
        ("dstate", ctypes.c_int64),
        ("io_dtype", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("x", ctypes.c_void_p),
        ("dt", ctypes.c_void_p),
        ("A", ctypes.c_void_p),
        ("Bm", ctypes.c_void_p),
        ("Cm", ctypes.c_void_p),
        ("D", ctypes.c_void_p),
        ("state", ctypes.c_void_p),
        ("y", ctypes.c_void_p),
    ]


class SsdFwdMimoArgs(ctypes.Structure):
    _fields_ = [
        ("base", SsdFwdArgs),
        ("rank", ctypes.c_int64),
    ]


class SsdFwdRotArgs(ctypes.Structure):
    _fields_ = [
        ("base", SsdFwdArgs),
        ("theta", ctypes.c_void_p),
        ("init_state_im", ctypes.c_void_p),
        ("final_state_im", ctypes.c_void_p),
    ]


class SsdBwdArgs(ctypes.Structure):
    _fields_ = [
        ("fwd", SsdFwdArgs),
        ("dy", ctypes.c_void_p),
        ("dfinal", ctypes.c_void_p),
        ("dx", ctypes.c_void_p),
        ("ddt", ctypes.c_void_p),
        ("dA", ctypes.c_void_p),
        ("dBm", ctypes.c_void_p),
        ("dCm", ctypes.c_void_p),
        ("dD", ctypes.c_void_p),
        ("dinit", ctypes.c_void_p),
    ]


_lock = threading.Lock()
_lib = None

_VP = ctypes.c_void_p
_ARGS_P = ctypes.POINTER(SsdFwdArgs)

# name -> (restype, argtypes); every symbol include/ssd.h declares.
SIGNATURES = {
    "ssd_abi_version": (ctypes.c_int, []),
    "ssd_fwd_workspace_size": (ctypes.c_size_t, [_ARGS_P]),
    "ssd_fwd": (ctypes.c_int, [_ARGS_P, _VP]),
    "ssd_fwd_noalloc": (ctypes.c_int, [_ARGS_P, _VP]),
    "ssd_fwd_noalloc_status": (ctypes.c_int, [_VP]),
    "ssd_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "ssd_last_error_message": (ctypes.c_char_p, []),
    "ssd_workspace_status": (ctypes.c_int, [_VP, _VP]),
    "ssd_fwd_host_workspace_size": (ctypes.c_size_t, [_ARGS_P]),
    "ssd_fwd_host": (ctypes.c_int, [_ARGS_P, _VP]),
    "ssd_fwd_ex_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(SsdFwdExArgs)]),
    "ssd_fwd_ex": (ctypes.c_int, [ctypes.POINTER(SsdFwdExArgs), _VP]),
    "ssd_step": (ctypes.c_int, [ctypes.POINTER(SsdStepArgs), _VP]),
    "ssd_fwd_mimo_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(SsdFwdMimoArgs)]),
    "ssd_fwd_mimo": (ctypes.c_int, [ctypes.POINTER(SsdFwdMimoArgs), _VP]),
    "ssd_fwd_rot_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(SsdFwdRotArgs)]),
    "ssd_fwd_rot": (ctypes.c_int, [ctypes.POINTER(SsdFwdRotArgs), _VP]),
    "ssd_bwd_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(SsdBwdArgs)]),
    "ssd_bwd": (ctypes.c_int, [ctypes.POINTER(SsdBwdArgs), _VP]),
    "ssd_chunk_cumsum": (ctypes.c_int, [_ARGS_P, ctypes.c_int64, _VP, _VP, _VP]),
    "ssd_chunk_state": (ctypes.c_int, [_ARGS_P, ctypes.c_int64, _VP, _VP, _VP, _VP]),
    "ssd_state_passing": (ctypes.c_int, [_ARGS_P, ctypes.c_int64, _VP, _VP, _VP]),
    "ssd_chunk_scan": (ctypes.c_int, [_ARGS_P, ctypes.c_int64, _VP, _VP, _VP, _VP]),
}


def lib():
    """The loaded library (loads it on first use; raises if it is not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -m ssd_scan_fwd_b300.build` "
                    "(there is no fallback implementation)")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


class SsdError(RuntimeError):
    def __init__(self, status: int, where: str):
        L = lib()
        msg = L.ssd_status_string(status).decode()
        detail = L.ssd_last_error_message().decode()
        super().__init__(f"{where}: {msg}" + (f" ({detail})" if detail else ""))
        self.status = status


def check(status: int, where: str) -> None:
    if status != SSD_OK:
        raise SsdError(status, where)
