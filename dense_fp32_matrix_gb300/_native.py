"""ctypes loader for libdfm_sgemm.so (the C ABI in include/dfm_sgemm.h).

There is no fallback: if the library is missing or cannot be loaded, every
entry point raises. Build it with ``python -m dense_fp32_matrix_gb300.build``
or ``__graft_entry__.build()``.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

LIB_PATH = _build.LIB

_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_int = ctypes.c_int

_SIGNATURES = {
    "sgemm": ([_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp], _int),
    "sgemm_path": ([_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp,
                    _int], _int),
    "sgemm_plan": ([_i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_uint64,
                    ctypes.c_uint64, ctypes.c_uint64, ctypes.POINTER(_int)],
                   _int),
    "sgemm_ex": ([_int, _int, _i64, _i64, _i64, ctypes.c_float, _vp, _i64,
                  _vp, _i64, ctypes.c_float, _vp, _i64, _vp], _int),
    "sgemm_ex_path": ([_int, _int, _i64, _i64, _i64, ctypes.c_float, _vp,
                       _i64, _vp, _i64, ctypes.c_float, _vp, _i64, _vp, _int],
                      _int),
    "sgemm_plan_ex": ([_int, _int, _i64, _i64, _i64, _i64, _i64, _i64,
                       ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                       ctypes.POINTER(_int)], _int),
    "sgemm_strided_batched": ([_int, _int, _i64, _i64, _i64, ctypes.c_float,
                               _vp, _i64, _i64, _vp, _i64, _i64,
                               ctypes.c_float, _vp, _i64, _i64, _i64, _vp],
                              _int),
    "sgemm_strided_batched_path": ([_int, _int, _i64, _i64, _i64,
                                    ctypes.c_float, _vp, _i64, _i64, _vp,
                                    _i64, _i64, ctypes.c_float, _vp, _i64,
                                    _i64, _i64, _vp, _int], _int),
    "sgemm_noalloc": ([_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp],
                      _int),
    "sgemm_host": ([_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp,
                    _vp, _vp, _vp], _int),
    "sgemm_set_math_mode": ([_int], _int),
    "sgemm_watchdog_status": ([ctypes.POINTER(_int)], _int),
    "sgemm_watchdog_selftest": ([_vp, _i64], _int),
    "sgemm_workspace_info": ([ctypes.POINTER(_int), ctypes.POINTER(_i64)],
                             _int),
    "sgemm_status_string": ([_int], ctypes.c_char_p),
    "sgemm_path_name": ([_int], ctypes.c_char_p),
    "sgemm_version": ([], _int),
    "sgemm_launch_count": ([], ctypes.c_uint64),
}


class NativeLibraryMissing(ImportError):
    pass


def lib():
    """The loaded library (loads on first use; raises if it is not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise NativeLibraryMissing(
                    "%s is not built; run `python -m dense_fp32_matrix_gb300."
                    "build` (needs nvcc)" % LIB_PATH)
            handle = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in _SIGNATURES.items():
                f = getattr(handle, name)
                f.argtypes = args
                f.restype = res
            _lib = handle
    return _lib


def exported_symbols():
    return list(_SIGNATURES)
