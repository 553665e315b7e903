"""fp64 CPU oracle for C = A * B (row-major fp32 inputs).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm may import this package. The CUDA
product path neither imports it nor shares code with it.

Thin ctypes wrapper over ``sgemm_oracle.c`` (see its header for the formula
and the passages it follows). Results come back in fp64; callers round to
fp32 once when they need the fp32 result.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build as _build

__all__ = ["gemm", "gemm_ex", "gemm_rows", "gemm_entries", "num_threads",
           "round_fp32", "bound", "ORACLE_LIB"]

_lock = threading.Lock()
_lib = None
ORACLE_LIB = _build.LIB

_i64 = ctypes.c_int64
_fp = ctypes.POINTER(ctypes.c_float)
_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int64)


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            lib = ctypes.CDLL(path)
            sig = [_i64, _i64, _i64, _fp, _i64, _fp, _i64, _dp, _i64, _dp, _i64]
            for name in ("oracle_gemm_inner", "oracle_gemm_outer"):
                f = getattr(lib, name)
                f.argtypes = sig
                f.restype = ctypes.c_int
            lib.oracle_gemm_rows.argtypes = [_i64, _i64, _i64, _fp, _i64, _fp,
                                             _i64, _ip, _i64, _dp, _dp]
            lib.oracle_gemm_rows.restype = ctypes.c_int
            lib.oracle_gemm_entries.argtypes = [_i64, _i64, _i64, _fp, _i64,
                                                _fp, _i64, _ip, _ip, _i64,
                                                _dp, _dp]
            lib.oracle_gemm_entries.restype = ctypes.c_int
            lib.oracle_gemm_ex.argtypes = [ctypes.c_int, ctypes.c_int, _i64,
                                           _i64, _i64, ctypes.c_double, _fp,
                                           _i64, _fp, _i64, ctypes.c_double,
                                           _fp, _i64, _dp, _i64, _dp, _i64]
            lib.oracle_gemm_ex.restype = ctypes.c_int
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _fptr(a):
    if a is None:
        return None
    assert a.dtype == np.float32 and a.flags.c_contiguous
    return a.ctypes.data_as(_fp)


def _dptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def _operands(A, B, M, N, K, lda, ldb):
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    if M is None:
        M, K = A.shape
    if N is None:
        N = B.shape[1]
    if lda is None:
        lda = A.shape[1] if A.ndim == 2 else max(K, 1)
    if ldb is None:
        ldb = B.shape[1] if B.ndim == 2 else max(N, 1)
    return A, B, int(M), int(N), int(K), int(lda), int(ldb)


def gemm(A, B, M=None, N=None, K=None, lda=None, ldb=None, order="outer",
         with_abs=True):
    """Full product in fp64. Returns ``(C, S)`` (S is None when not asked).

    ``A``/``B`` hold row-major fp32 data with leading dimensions lda/ldb
    (taken from the array shapes when omitted). ``order`` is "outer" (i-k-j)
    or "inner" (i-j-k).
    """
    A, B, M, N, K, lda, ldb = _operands(A, B, M, N, K, lda, ldb)
    C = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64) if with_abs else None
    fn = {"outer": _load().oracle_gemm_outer,
          "inner": _load().oracle_gemm_inner}[order]
    rc = fn(M, N, K, _fptr(A), lda, _fptr(B), ldb, _dptr(C), max(N, 1),
            _dptr(S), max(N, 1))
    if rc != 0:
        raise ValueError("oracle rejected arguments (M=%d N=%d K=%d lda=%d "
                         "ldb=%d)" % (M, N, K, lda, ldb))
    return C, S


def gemm_ex(op_a, op_b, alpha, A, B, beta, C0, M, N, K, lda=None, ldb=None,
            ldc0=None):
    """``alpha * op(A) * op(B) + beta * C0`` in fp64; returns ``(C, S)``.

    ``op_a`` / ``op_b`` are "N" or "T". A is stored M x K ("N", ld >= K) or
    K x M ("T", ld >= M); B is stored K x N ("N", ld >= N) or N x K ("T",
    ld >= K). C0 (M x N, ld ``ldc0``) is not read when beta == 0, A and B
    are not read when alpha == 0 (pass None for unread operands).
    """
    oa, ob = {"N": 0, "T": 1}[op_a], {"N": 0, "T": 1}[op_b]
    M, N, K = int(M), int(N), int(K)

    def prep(X, cols):
        if X is None:
            return None, max(cols, 1)
        X = np.ascontiguousarray(X, dtype=np.float32)
        return X, max(X.shape[1] if X.ndim == 2 else cols, 1)
    A, lda_d = prep(A, M if oa else K)
    B, ldb_d = prep(B, K if ob else N)
    C0, ldc_d = prep(C0, N)
    C = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_ex(oa, ob, M, N, K, float(alpha), _fptr(A),
                                int(lda or lda_d), _fptr(B), int(ldb or ldb_d),
                                float(beta), _fptr(C0), int(ldc0 or ldc_d),
                                _dptr(C), max(N, 1), _dptr(S), max(N, 1))
    if rc != 0:
        raise ValueError("oracle rejected arguments")
    return C, S


def gemm_rows(A, B, rows, M=None, N=None, K=None, lda=None, ldb=None):
    """Rows ``rows`` of C and S in fp64, shape (len(rows), N) each."""
    A, B, M, N, K, lda, ldb = _operands(A, B, M, N, K, lda, ldb)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    C = np.zeros((len(r), N), dtype=np.float64)
    S = np.zeros((len(r), N), dtype=np.float64)
    rc = _load().oracle_gemm_rows(M, N, K, _fptr(A), lda, _fptr(B), ldb,
                                  r.ctypes.data_as(_ip), len(r), _dptr(C),
                                  _dptr(S))
    if rc != 0:
        raise ValueError("oracle rejected arguments")
    return C, S


def gemm_entries(A, B, ii, jj, M=None, N=None, K=None, lda=None, ldb=None):
    """Entries C[ii[e], jj[e]] and S[ii[e], jj[e]] in fp64."""
    A, B, M, N, K, lda, ldb = _operands(A, B, M, N, K, lda, ldb)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    assert ii.shape == jj.shape
    c = np.zeros(ii.shape, dtype=np.float64)
    s = np.zeros(ii.shape, dtype=np.float64)
    rc = _load().oracle_gemm_entries(M, N, K, _fptr(A), lda, _fptr(B), ldb,
                                     ii.ctypes.data_as(_ip),
                                     jj.ctypes.data_as(_ip), len(ii),
                                     _dptr(c), _dptr(s))
    if rc != 0:
        raise ValueError("oracle rejected arguments")
    return c, s


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def round_fp32(C64):
    """The oracle's fp32 result: the fp64 sum rounded once to nearest."""
    return np.asarray(C64, dtype=np.float64).astype(np.float32)


def bound(S64, rel=1e-4, abs_=1e-6):
    """Per-element tolerance |C_gpu - C_oracle| <= rel * S + abs."""
    return rel * np.asarray(S64, dtype=np.float64) + abs_
