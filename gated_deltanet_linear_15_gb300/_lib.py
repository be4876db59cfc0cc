"""ctypes view of the C ABI declared in include/gdn.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

GDN_BF16, GDN_FP32 = 0, 1
GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_WORKSPACE, GDN_ERR_CUDA = 0, 1, 2, 3, 4
GDN_ERR_TIMEOUT, GDN_ERR_NUMERIC = 5, 6
GDN_L2NORM_QK, GDN_SP_OFF, GDN_WINDOW_OFF, GDN_SP_SINGLE_LAUNCH = 1, 2, 4, 8
GDN_DEBUG_WAIT_TIMEOUT = 0x80000000
GDN_DEBUG_PEER_TIMEOUT = 0x40000000
GDN_STATIC_SCRATCH_BYTES = 16 << 20

# every symbol include/gdn.h declares
EXPORTS = ("gdn_fwd_workspace_size", "gdn_bwd_workspace_size", "gdn_chunk_fwd", "gdn_chunk_fwd_static",
           "gdn_chunk_bwd", "gdn_saved_size", "gdn_bwd_saved_workspace_size", "gdn_chunk_fwd_save",
           "gdn_chunk_bwd_saved", "gdn_recurrent_fwd",
           "gdn_get_device_status", "gdn_device_status_code", "gdn_plan_query", "gdn_plan_estimate", "gdn_profile_enable", "gdn_profile_report", "gdn_profile_only",
           "gdn_status_string", "gdn_last_error_string")


class GdnShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("Dk", ctypes.c_int), ("Dv", ctypes.c_int),
                ("cu_seqlens", ctypes.c_void_p), ("num_seqs", ctypes.c_int),
                ("dtype", ctypes.c_int), ("scale", ctypes.c_float), ("flags", ctypes.c_uint),
                ("seg_chunks", ctypes.c_int), ("seg_first", ctypes.c_int),
                ("reserved", ctypes.c_int * 2)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load():
    """Load libgdn.so.  Raises if it has not been built: there is no fallback."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build the CUDA library first "
                              "(gated_deltanet_linear_15_gb300.build.build() or __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        P, S = ctypes.c_void_p, ctypes.POINTER(GdnShape)
        lib.gdn_fwd_workspace_size.argtypes = [S]
        lib.gdn_fwd_workspace_size.restype = ctypes.c_size_t
        lib.gdn_bwd_workspace_size.argtypes = [S]
        lib.gdn_bwd_workspace_size.restype = ctypes.c_size_t
        lib.gdn_chunk_fwd.argtypes = [S, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
        lib.gdn_chunk_fwd.restype = ctypes.c_int
        lib.gdn_chunk_fwd_static.argtypes = [S, P, P, P, P, P, P, P, P, P]
        lib.gdn_chunk_fwd_static.restype = ctypes.c_int
        lib.gdn_chunk_bwd.argtypes = [S, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
        lib.gdn_chunk_bwd.restype = ctypes.c_int
        lib.gdn_saved_size.argtypes = [S]
        lib.gdn_saved_size.restype = ctypes.c_size_t
        lib.gdn_bwd_saved_workspace_size.argtypes = [S]
        lib.gdn_bwd_saved_workspace_size.restype = ctypes.c_size_t
        lib.gdn_chunk_fwd_save.argtypes = [S, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P, ctypes.c_size_t, P]
        lib.gdn_chunk_fwd_save.restype = ctypes.c_int
        lib.gdn_chunk_bwd_saved.argtypes = [S, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P,
                                            ctypes.c_size_t, P]
        lib.gdn_chunk_bwd_saved.restype = ctypes.c_int
        lib.gdn_recurrent_fwd.argtypes = [S, P, P, P, P, P, P, P, P, P]
        lib.gdn_recurrent_fwd.restype = ctypes.c_int
        lib.gdn_get_device_status.argtypes = [S, P, P]
        lib.gdn_get_device_status.restype = ctypes.c_int
        lib.gdn_device_status_code.argtypes = [ctypes.c_int]
        lib.gdn_device_status_code.restype = ctypes.c_int
        lib.gdn_plan_query.argtypes = [S, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                                       ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
        lib.gdn_plan_query.restype = ctypes.c_int
        lib.gdn_plan_estimate.argtypes = [S, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
        lib.gdn_plan_estimate.restype = ctypes.c_int
        lib.gdn_profile_enable.argtypes = [ctypes.c_int]
        lib.gdn_profile_enable.restype = ctypes.c_int
        lib.gdn_profile_report.argtypes = [ctypes.c_char_p, ctypes.c_size_t, ctypes.c_int]
        lib.gdn_profile_report.restype = ctypes.c_int
        lib.gdn_profile_only.argtypes = [ctypes.c_char_p]
        lib.gdn_profile_only.restype = ctypes.c_int
        lib.gdn_status_string.argtypes = [ctypes.c_int]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_last_error_string.argtypes = []
        lib.gdn_last_error_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def last_error() -> str:
    return load().gdn_last_error_string().decode()
