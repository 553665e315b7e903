"""sgemm_noalloc: the entry point for callers that cannot allocate device
memory when they multiply (memory owned by another allocator, no implicit
device synchronisation allowed, no allocation after start-up). Its stream-K
scratch is a fixed device array inside the library.

Checked through the C ABI against sgemm(), the regular entry point, on two
calls in a row (the scratch keeps the previous call's contents). Collected
last on purpose: if it fails, a run that stops at the first failure has run
everything else already; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest

import matgen

pytestmark = pytest.mark.gpu

REL, ABS = 1e-4, 1e-6


@pytest.fixture(scope="module")
def lib():
    from dense_fp32_matrix_gb300 import _native, build
    build.build()
    L = _native.lib()
    return L


def _call(fn, M, N, K, A, B, C, stream):
    rc = fn(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N, stream)
    assert rc == 0, rc


@pytest.fixture(params=["ffma", "auto"])
def math_mode(request, lib):
    # "ffma" routes aligned shapes to the stream-K kernel, the one that uses
    # the fixed scratch; "auto" to the tensor-core kernel (no scratch).
    modes = {"auto": 0, "ffma": 1}
    previous = lib.sgemm_set_math_mode(modes[request.param])
    yield request.param
    lib.sgemm_set_math_mode(previous)


@pytest.mark.parametrize("M,N,K,kind", [
    (1000, 1100, 700, "uniform"),
    (2048, 2048, 2048, "integers"),
    (4096, 4096, 1024, "uniform"),
    (300, 200, 20, "uniform"),
    (127, 129, 33, "integers"),   # unaligned: a path without scratch
])
def test_noalloc_matches_sgemm_on_two_calls(lib, math_mode, M, N, K, kind):
    import torch
    A_h = matgen.KINDS[kind](17, matgen.MATRIX_A, M, K)
    B_h = matgen.KINDS[kind](17, matgen.MATRIX_B, K, N)
    A = torch.from_numpy(A_h).cuda()
    B = torch.from_numpy(B_h).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    C_ref = torch.empty((M, N), device="cuda")
    _call(lib.sgemm, M, N, K, A, B, C_ref, stream)
    outs = []
    for _ in range(2):
        C = torch.full((M, N), float("nan"), device="cuda")
        _call(lib.sgemm_noalloc, M, N, K, A, B, C, stream)
        outs.append(C)
    torch.cuda.synchronize()
    site = ctypes.c_int(0)
    assert lib.sgemm_watchdog_status(ctypes.byref(site)) == 0
    ref = C_ref.cpu().numpy().astype(np.float64)
    S = np.abs(A_h.astype(np.float64)) @ np.abs(B_h.astype(np.float64))
    for C in outs:
        got = C.cpu().numpy().astype(np.float64)
        if kind == "integers":
            assert np.array_equal(got, ref)
        else:
            assert np.isfinite(got).all()
            assert np.all(np.abs(got - ref) <= REL * S + ABS)
    # the scratch is reused: the second call gives the same bits as the first
    assert torch.equal(outs[0], outs[1])


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    # 16385 output tiles of 128 x 128 is one over the limit; rejected on the
    # host before anything is enqueued (the pointers are never touched).
    M, N = 128 * 16385, 128
    fake = 1 << 40
    rc = lib.sgemm_noalloc(M, N, 4, fake, 4, fake + (1 << 36), N,
                           fake + (1 << 38), N, None)
    assert rc == -9   # SGEMM_ERR_TOO_LARGE
