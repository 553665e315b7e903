"""GB300 (sm_103a) FP32 matrix product C = A * B, row-major fp32.

Thin Python binding over the C ABI of ``libdfm_sgemm.so``
(``include/dfm_sgemm.h``): the functions below carry the same names and
arguments and only marshal them; every step of the product runs in the CUDA
kernels. PyTorch is used only for device memory and streams, in ``matmul``.
"""
from __future__ import annotations

import ctypes

from . import _native

__all__ = [
    "SgemmError", "sgemm", "sgemm_path", "sgemm_plan", "sgemm_host",
    "sgemm_ex", "sgemm_plan_ex", "sgemm_strided_batched", "OPS",
    "sgemm_noalloc", "sgemm_set_math_mode", "MATH",
    "sgemm_watchdog_status", "sgemm_watchdog_selftest",
    "sgemm_workspace_info", "sgemm_status_string", "sgemm_path_name", "sgemm_version", "sgemm_launch_count", "matmul",
    "PATHS", "STATUS",
]

STATUS = {
    "SGEMM_OK": 0, "SGEMM_ERR_INVALID_VALUE": -1, "SGEMM_ERR_NULL_POINTER": -2,
    "SGEMM_ERR_UNSUPPORTED_DEVICE": -3, "SGEMM_ERR_LAUNCH": -4,
    "SGEMM_ERR_WATCHDOG": -5, "SGEMM_ERR_OVERLAP": -6, "SGEMM_ERR_CUDA": -7,
    "SGEMM_ERR_PATH": -8, "SGEMM_ERR_TOO_LARGE": -9,
}
MATH = {"auto": 0, "ffma": 1}
PATHS = {"auto": 0, "tiled_tma": 1, "tiled_ldg": 2, "gemv_row": 3,
         "gemv_col": 4, "naive": 5, "tf32x3": 6, "tf32x3_pair": 7,
         "small": 8}


class SgemmError(RuntimeError):
    def __init__(self, status: int, what: str = "sgemm"):
        self.status = int(status)
        super().__init__("%s failed: %s (%d)" % (
            what, sgemm_status_string(status), status))


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise SgemmError(rc, what)


def _ptr(x) -> int | None:
    """Device/host address of an int or a tensor-like with data_ptr()."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _path(path) -> int:
    if isinstance(path, str):
        return PATHS[path]
    return int(path)


def sgemm(M, N, K, A, lda, B, ldb, C, ldc, stream=None) -> None:
    """C[i*ldc+j] = sum_k A[i*lda+k] * B[k*ldb+j] on ``stream`` (async)."""
    _check(_native.lib().sgemm(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C),
                               ldc, _stream(stream)), "sgemm")


def sgemm_path(M, N, K, A, lda, B, ldb, C, ldc, stream=None, path="auto"):
    """As ``sgemm`` but on the named kernel path (see ``PATHS``)."""
    _check(_native.lib().sgemm_path(M, N, K, _ptr(A), lda, _ptr(B), ldb,
                                    _ptr(C), ldc, _stream(stream),
                                    _path(path)), "sgemm_path")


OPS = {"N": 0, "T": 1}


def _op(op) -> int:
    return OPS[op] if isinstance(op, str) else int(op)


def sgemm_ex(op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
             stream=None, path="auto") -> None:
    """C = alpha * op(A) * op(B) + beta * C on ``stream`` (async).

    ``op_a`` / ``op_b`` are "N" (as stored) or "T" (stored transposed: A as
    K x M, B as N x K). beta == 0 leaves C unread; alpha == 0 leaves A and B
    unread. ``path`` forces a kernel path like ``sgemm_path``.
    """
    lib = _native.lib()
    if path == "auto":
        rc = lib.sgemm_ex(_op(op_a), _op(op_b), M, N, K, float(alpha),
                          _ptr(A), lda, _ptr(B), ldb, float(beta), _ptr(C),
                          ldc, _stream(stream))
    else:
        rc = lib.sgemm_ex_path(_op(op_a), _op(op_b), M, N, K, float(alpha),
                               _ptr(A), lda, _ptr(B), ldb, float(beta),
                               _ptr(C), ldc, _stream(stream), _path(path))
    _check(rc, "sgemm_ex")


def sgemm_plan_ex(op_a, op_b, M, N, K, lda, ldb, ldc, a_addr, b_addr,
                  c_addr) -> str:
    """Name of the kernel path ``sgemm_ex`` would take (host-only)."""
    out = ctypes.c_int(-1)
    _check(_native.lib().sgemm_plan_ex(_op(op_a), _op(op_b), M, N, K, lda,
                                       ldb, ldc, a_addr, b_addr, c_addr,
                                       ctypes.byref(out)), "sgemm_plan_ex")
    return sgemm_path_name(out.value)


def sgemm_strided_batched(op_a, op_b, M, N, K, alpha, A, lda, stride_a, B,
                          ldb, stride_b, beta, C, ldc, stride_c, batch,
                          stream=None, path="auto") -> None:
    """``batch`` products C_b = alpha op(A_b) op(B_b) + beta C_b with X_b =
    X + b * stride_x (floats; stride 0 shares the operand) on ``stream``."""
    lib = _native.lib()
    args = (_op(op_a), _op(op_b), M, N, K, float(alpha), _ptr(A), lda,
            stride_a, _ptr(B), ldb, stride_b, float(beta), _ptr(C), ldc,
            stride_c, batch, _stream(stream))
    if path == "auto":
        rc = lib.sgemm_strided_batched(*args)
    else:
        rc = lib.sgemm_strided_batched_path(*args, _path(path))
    _check(rc, "sgemm_strided_batched")


def sgemm_noalloc(M, N, K, A, lda, B, ldb, C, ldc, stream=None) -> None:
    """As ``sgemm`` but never allocates device memory (fixed scratch)."""
    _check(_native.lib().sgemm_noalloc(M, N, K, _ptr(A), lda, _ptr(B), ldb,
                                       _ptr(C), ldc, _stream(stream)),
           "sgemm_noalloc")


def sgemm_set_math_mode(mode) -> str:
    """Process-wide math mode ("auto" or "ffma"); returns the previous one."""
    m = MATH[mode] if isinstance(mode, str) else int(mode)
    rc = int(_native.lib().sgemm_set_math_mode(m))
    if rc < 0:
        raise SgemmError(rc, "sgemm_set_math_mode")
    return {v: k for k, v in MATH.items()}[rc]


def sgemm_plan(M, N, K, lda, ldb, ldc, a_addr, b_addr, c_addr) -> str:
    """Name of the path ``sgemm`` would take (host-only decision)."""
    out = ctypes.c_int(-1)
    _check(_native.lib().sgemm_plan(M, N, K, lda, ldb, ldc, a_addr, b_addr,
                                    c_addr, ctypes.byref(out)), "sgemm_plan")
    return sgemm_path_name(out.value)


def sgemm_host(M, N, K, hA, lda, hB, ldb, hC, ldc, dA, dB, dC,
               stream=None) -> None:
    """Host matrices in, host C out, through device staging buffers."""
    _check(_native.lib().sgemm_host(M, N, K, _ptr(hA), lda, _ptr(hB), ldb,
                                    _ptr(hC), ldc, _ptr(dA), _ptr(dB),
                                    _ptr(dC), _stream(stream)), "sgemm_host")


def sgemm_watchdog_status() -> tuple[int, int]:
    """(status, site) of the bounded device waits; reads and clears."""
    site = ctypes.c_int(0)
    rc = _native.lib().sgemm_watchdog_status(ctypes.byref(site))
    return rc, site.value


def sgemm_watchdog_selftest(stream=None, timeout_ns=50_000_000) -> int:
    return int(_native.lib().sgemm_watchdog_selftest(_stream(stream),
                                                     int(timeout_ns)))


def sgemm_workspace_info() -> tuple[int, int]:
    """(count, bytes) of the workspaces held on the current device."""
    count = ctypes.c_int(0)
    nbytes = ctypes.c_int64(0)
    _check(_native.lib().sgemm_workspace_info(ctypes.byref(count),
                                              ctypes.byref(nbytes)),
           "sgemm_workspace_info")
    return count.value, nbytes.value


def sgemm_status_string(status: int) -> str:
    return _native.lib().sgemm_status_string(int(status)).decode()


def sgemm_path_name(path: int) -> str:
    return _native.lib().sgemm_path_name(int(path)).decode()


def sgemm_version() -> int:
    return int(_native.lib().sgemm_version())


def sgemm_launch_count() -> int:
    """Kernel launches the library has issued in this process."""
    return int(_native.lib().sgemm_launch_count())


def matmul(A, B, out=None, path="auto", stream=None):
    """torch convenience: ``out = A @ B`` for fp32 CUDA tensors.

    A (M x K) and B (K x N) need unit column stride (row-major with any row
    pitch); ``out`` (M x N) likewise, allocated with torch when omitted.
    """
    import torch
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("shape mismatch: %s @ %s" % (tuple(A.shape),
                                                     tuple(B.shape)))
    for name, t in (("A", A), ("B", B)):
        if t.dtype != torch.float32 or not t.is_cuda:
            raise TypeError("%s must be a float32 CUDA tensor" % name)
        if t.shape[1] > 1 and t.stride(1) != 1:
            raise ValueError("%s needs unit column stride" % name)
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if out.shape != (M, N) or (N > 1 and out.stride(1) != 1):
        raise ValueError("out must be (M, N) with unit column stride")
    def pitch(t, rows, cols):
        if rows <= 1:
            return max(cols, 1)
        if t.stride(0) < cols:
            raise ValueError("row pitch below the row width")
        return t.stride(0)
    lda, ldb, ldc = pitch(A, M, K), pitch(B, K, N), pitch(out, M, N)
    sgemm_path(M, N, K, A, lda, B, ldb, out, ldc, stream, path)
    return out
