"""sgemm_noalloc: the entry point for callers that cannot allocate device
memory when they multiply (memory owned by another allocator, no implicit
device synchronisation allowed, no allocation after start-up). Its stream-K
scratch is a fixed device array inside the library.

Checked through the C ABI against the CPU oracle and against sgemm(), the
regular entry point, on two calls in a row (the scratch keeps the previous
call's contents, so the second call must not depend on it). Collected last
on purpose: if it fails, a run that stops at the first failure has run
everything else already; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest

import matgen
import oracle
from gpu_util import FULL_CHECK_MAX_MNK, compare, sample_indices

pytestmark = pytest.mark.gpu

REL, ABS = 1e-4, 1e-6
TOO_LARGE = -9


@pytest.fixture(scope="module")
def lib():
    from dense_fp32_matrix_gb300 import _native, build
    build.build()
    L = _native.lib()
    return L


def _call(fn, M, N, K, A, B, C, stream):
    rc = fn(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N, stream)
    assert rc == 0, rc


def _check_oracle(kind, got, A_h, B_h, M, N, K, what):
    if M * N * K <= FULL_CHECK_MAX_MNK:
        ref, S = oracle.gemm(A_h, B_h)
        compare(kind, got, ref, S, what)
        return
    rows, ii, jj = sample_indices(M, N)
    ref, S = oracle.gemm_rows(A_h, B_h, rows)
    compare(kind, got[rows], ref, S, what + " rows")
    c, s = oracle.gemm_entries(A_h, B_h, ii, jj)
    compare(kind, got[ii, jj], c, s, what + " entries")


@pytest.fixture(params=["ffma", "auto"])
def math_mode(request, lib):
    # "ffma" routes aligned shapes to the stream-K kernel, the one that uses
    # the fixed scratch; "auto" to the tensor-core kernels (whole tiles, no
    # split k: no scratch).
    modes = {"auto": 0, "ffma": 1}
    previous = lib.sgemm_set_math_mode(modes[request.param])
    yield request.param
    lib.sgemm_set_math_mode(previous)


@pytest.mark.parametrize("M,N,K,kind", [
    (1000, 1100, 700, "uniform"),
    (2048, 2048, 2048, "integers"),
    (4096, 4096, 1024, "uniform"),
    # 9 x 9 pair tiles on 76 clusters: sgemm gives the tail to stream-K, the
    # scratch-free call runs whole tiles only (a second wave of 5 tiles)
    (2304, 2304, 2048, "uniform"),
    # few short-k tiles: sgemm splits k over idle SMs, this call does not
    (1024, 1024, 640, "integers"),
    (300, 200, 20, "uniform"),
    (127, 129, 33, "integers"),   # unaligned: a path without scratch
    # rows not 16-byte aligned and at least 2^32 multiply-adds: sgemm
    # repacks both operands into its workspace (tensor path, or the TMA
    # tile kernel in ffma mode); this call takes the any-layout kernel
    (2055, 2057, 1023, "integers"),
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
    for n, C in enumerate(outs):
        _check_oracle(kind, C.cpu().numpy(), A_h, B_h, M, N, K,
                      "noalloc call %d %s %dx%dx%d" % (n, math_mode, M, N, K))
    # against the regular entry point: the same bits on integer data, the
    # accuracy bound on float data (another split may change the last bits)
    ref = C_ref.cpu().numpy().astype(np.float64)
    S = np.abs(A_h.astype(np.float64)) @ np.abs(B_h.astype(np.float64))
    got = outs[0].cpu().numpy().astype(np.float64)
    if kind == "integers":
        assert np.array_equal(got, ref)
    else:
        assert np.all(np.abs(got - ref) <= 2 * (REL * S + ABS))
    # the scratch is reused: the second call gives the same bits as the first
    assert torch.equal(outs[0], outs[1])


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    # In the CUDA-core mode an aligned product takes the stream-K kernel,
    # whose tile counters live in the scratch: 16385 output tiles of
    # 256 x 128 is one over the limit, rejected on the host before anything
    # is enqueued. The buffers are real (2.1 GB for C) and C is checked
    # untouched, so a regression shows up as a failed assertion.
    import torch
    M, N, K = 256 * 16385, 128, 4
    A = torch.zeros((M, K), device="cuda")
    B = torch.zeros((K, N), device="cuda")
    C = torch.full((M, N), 7.0, device="cuda")
    torch.cuda.synchronize()
    previous = lib.sgemm_set_math_mode(1)
    try:
        rc = lib.sgemm_noalloc(M, N, K, A.data_ptr(), K, B.data_ptr(), N,
                               C.data_ptr(), N, None)
    finally:
        lib.sgemm_set_math_mode(previous)
    torch.cuda.synchronize()
    assert rc == TOO_LARGE
    assert bool((C[::4096] == 7.0).all())


def test_noalloc_limit_spares_paths_without_scratch(lib):
    # A vector product as wide as 16385 tiles uses no scratch: it runs.
    import torch
    M, N, K = 1, 128 * 16385, 64
    a_h = matgen.uniform(18, matgen.MATRIX_A, M, K)
    B_h = matgen.uniform(18, matgen.MATRIX_B, K, N)
    a = torch.from_numpy(a_h).cuda()
    B = torch.from_numpy(B_h).cuda()
    c = torch.full((M, N), float("nan"), device="cuda")
    _call(lib.sgemm_noalloc, M, N, K, a, B, c, None)
    torch.cuda.synchronize()
    ref, S = oracle.gemm(a_h, B_h)
    compare("uniform", c.cpu().numpy(), ref, S, "noalloc wide vector")
