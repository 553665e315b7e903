"""Parity of the CUDA path with the CPU oracle, through the C ABI.

Bit-exact on integer-valued inputs; |C - C_oracle| <= 1e-4 * S + 1e-6 per
element otherwise (S = sum_k |A_ik B_kj|). Full comparison for shapes up to
2^33 multiply-adds, else 64 full rows plus 4096 sampled entries."""
import itertools

import numpy as np
import pytest

import matgen
import oracle
from matgen.workloads import WORKLOADS
from gpu_util import compare, run_case, upload, download_c, SENTINEL_BITS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    # This module covers the CUDA-core fp32 FMA paths: "auto" here resolves
    # to them (the tensor-core path has its own module).
    import dense_fp32_matrix_gb300 as dfm
    from dense_fp32_matrix_gb300 import build
    build.build()
    previous = dfm.sgemm_set_math_mode("ffma")
    yield
    dfm.sgemm_set_math_mode(previous)


@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w["name"])
def test_workload(w):
    run_case(w["M"], w["N"], w["K"], w["kind"], w["seed"])


def test_misaligned_large_product_takes_the_tma_kernel_on_copies():
    # From 2^32 multiply-adds, operands TMA cannot map (here: bases off 16
    # bytes, odd row strides) are repacked into the workspace and the
    # TMA-fed kernel runs; C keeps its own layout.
    import dense_fp32_matrix_gb300 as dfm
    M, N, K = 2055, 2057, 1023
    assert M * N * K >= 1 << 32
    a, b, c = 0x7f0000000004, 0x7f4000000008, 0x7f8000000000  # A, B off 16
    assert dfm.sgemm_plan(M, N, K, K, N, N, a, b, c) == "tiled_tma"
    assert dfm.sgemm_plan(2040, N, K, K, N, N, a, b, c) == "tiled_ldg"
    run_case(M, N, K, "integers", 5, offsets=(1, 3, 2))
    run_case(M, N, K, "uniform", 6, lda=K + 1, ldb=N + 2, ldc=N + 1)


# Shapes spanning several tiles plus a ragged tail in every dimension.
MULTI_TILE = [(300, 200, 20), (257, 383, 129), (128, 128, 32), (129, 257, 33),
              (640, 384, 96), (1000, 1000, 1000), (384, 256, 24)]


@pytest.mark.parametrize("path", ["auto", "tiled_ldg", "naive", "small"])
@pytest.mark.parametrize("mnk", MULTI_TILE, ids=str)
@pytest.mark.parametrize("kind", ["uniform", "integers"])
def test_multi_tile_paths(path, mnk, kind):
    run_case(*mnk, kind=kind, seed=sum(mnk), path=path)


@pytest.mark.parametrize("mnk", [(256, 256, 256), (384, 256, 24),
                                 (260, 132, 36), (1024, 512, 1000)], ids=str)
def test_tma_path_forced(mnk):
    # shapes whose K and N are multiples of 4 (16-byte TMA row strides)
    run_case(*mnk, kind="uniform", seed=5, path="tiled_tma")
    run_case(*mnk, kind="integers", seed=5, path="tiled_tma")


SIZES = (1, 2, 3, 4, 5, 7, 8, 9, 16, 17, 31, 33)


@pytest.mark.parametrize("path", ["auto", "tiled_ldg", "naive", "small"])
def test_brute_force_tiny_shapes(path):
    for M, N, K in itertools.product(SIZES, SIZES, SIZES):
        run_case(M, N, K, kind="integers", seed=M * 10000 + N * 100 + K,
                 path=path, check="full")


# (1, 1000, 777), (1, 20, 3), (1, 4096, 4096): 16-byte row strides, TMA
# kernel with a cluster k-split; (1, 17, 3), (1, 1, 5000): plain kernel.
@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (1, 1000, 777),
                                   (1, 1, 5000), (1, 17, 3), (1, 20, 3),
                                   (1, 4100, 65), (1, 64, 11008)])
def test_gemv_row(M, N, K):
    for kind in ("uniform", "integers"):
        run_case(M, N, K, kind=kind, seed=K, path="gemv_row")
    run_case(M, N, K, kind="uniform", seed=K, path="gemv_row", ldb=N + 5)


# K % 4 == 0 with ldb == 1: TMA kernel; otherwise the plain kernel.
# (8000, 1, 1000) and (8191, 1, 520): 500 and 512 blocks of 16 rows, more
# than one wave of 4-stage blocks and at most one of 3-stage blocks on
# 152 SMs, so the 3-stage ring runs (with a ragged last block of rows).
@pytest.mark.parametrize("M,N,K", [(4096, 1, 4096), (1000, 1, 777),
                                   (3, 1, 5000), (17, 1, 3), (1000, 1, 780),
                                   (33, 1, 260), (4097, 1, 11008),
                                   (8000, 1, 1000), (8191, 1, 520)])
def test_gemv_col(M, N, K):
    for kind in ("uniform", "integers"):
        run_case(M, N, K, kind=kind, seed=K, path="gemv_col")
    run_case(M, N, K, kind="uniform", seed=K, path="gemv_col", lda=K + 3,
             ldb=4)


@pytest.mark.parametrize("path", ["auto", "tiled_tma", "tiled_ldg"])
def test_pitch_padding_never_read_or_written(path):
    # NaN poison in the A/B padding, sentinel in the C padding and guards.
    run_case(300, 200, 64, "uniform", 9, lda=72, ldb=204, ldc=260, path=path)
    run_case(260, 132, 36, "integers", 9, lda=40, ldb=136, ldc=133, path=path)


@pytest.mark.parametrize("offsets", [(1, 0, 0), (0, 1, 0), (0, 0, 1),
                                     (3, 2, 1)])
def test_misaligned_pointers(offsets):
    run_case(257, 130, 68, "uniform", 4, offsets=offsets)
    run_case(64, 64, 64, "integers", 4, offsets=offsets)


def test_degenerate_sizes():
    # K = 0: C = 0 inside, padding untouched; M = 0 / N = 0: nothing written.
    import torch
    import dense_fp32_matrix_gb300 as dfm
    for (M, N, K, ldc) in [(5, 7, 0, 9), (0, 7, 3, 7), (5, 0, 3, 1)]:
        bufC, pC = upload(None, M, N, ldc, fill_bits=SENTINEL_BITS)
        dfm.sgemm(M, N, K, 0, max(K, 1), 0, max(N, 1), pC, ldc)
        torch.cuda.synchronize()
        C = download_c(bufC, M, N, ldc)
        assert C.shape == (M, N) and np.all(C == 0)
    run_case(1, 1, 1, "uniform", 1)
    run_case(2, 3, 1, "uniform", 1)   # K = 1: a rank-1 product, one rounding


def test_overlap_and_forced_path_errors():
    import torch
    import dense_fp32_matrix_gb300 as dfm
    buf = torch.zeros(4096, device="cuda")
    p = buf.data_ptr()
    with pytest.raises(dfm.SgemmError) as e:
        dfm.sgemm(8, 8, 8, p, 8, p + 4 * 1024, 8, p + 4 * 32, 8)
    assert e.value.status == dfm.STATUS["SGEMM_ERR_OVERLAP"]
    with pytest.raises(dfm.SgemmError) as e:
        dfm.sgemm_path(8, 8, 9, p, 9, p + 4 * 1024, 8, p + 4 * 2048, 8,
                       path="tiled_tma")
    assert e.value.status == dfm.STATUS["SGEMM_ERR_PATH"]
    with pytest.raises(dfm.SgemmError) as e:
        dfm.sgemm_path(2, 8, 8, p, 8, p + 4 * 1024, 8, p + 4 * 2048, 8,
                       path="gemv_row")
    assert e.value.status == dfm.STATUS["SGEMM_ERR_PATH"]


def test_nan_propagates_to_its_row_and_column():
    import torch
    import dense_fp32_matrix_gb300 as dfm
    A = torch.from_numpy(matgen.uniform(1, 0, 256, 256)).cuda()
    B = torch.from_numpy(matgen.uniform(1, 1, 256, 256)).cuda()
    A[7, 100] = float("nan")
    B[30, 200] = float("nan")
    C = dfm.matmul(A, B)
    torch.cuda.synchronize()
    nan = torch.isnan(C).cpu().numpy()
    assert nan[7].all() and nan[:, 200].all()
    nan[7] = False
    nan[:, 200] = False
    assert not nan.any()


def test_deterministic_and_stream_ordered():
    import torch
    import dense_fp32_matrix_gb300 as dfm
    A = torch.from_numpy(matgen.uniform(2, 0, 1000, 777)).cuda()
    B = torch.from_numpy(matgen.uniform(2, 1, 777, 999)).cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        C1 = dfm.matmul(A, B)
        C2 = dfm.matmul(A, B, stream=s)
    s.synchronize()
    assert torch.equal(C1, C2)


def test_host_buffers_entry_point():
    import torch
    import dense_fp32_matrix_gb300 as dfm
    M, N, K = 300, 260, 129
    A = matgen.uniform(8, 0, M, K)
    B = matgen.uniform(8, 1, K, N)
    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    hC = torch.full((M, N + 3), float("nan")).pin_memory()
    dA = torch.empty(M * K, device="cuda")
    dB = torch.empty(K * N, device="cuda")
    dC = torch.empty(M * N, device="cuda")
    dfm.sgemm_host(M, N, K, hA, K, hB, N, hC, N + 3, dA, dB, dC)
    torch.cuda.synchronize()
    ref64, S = oracle.gemm(A, B)
    compare("uniform", hC[:, :N].numpy(), ref64, S, "sgemm_host")
    assert torch.isnan(hC[:, N:]).all()
    # one pass of the same size: the same kernel, so the same bits
    ref = dfm.matmul(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
    torch.cuda.synchronize()
    assert torch.equal(hC[:, :N], ref.cpu())


def test_watchdog_timeout_is_reported_and_context_survives():
    import dense_fp32_matrix_gb300 as dfm
    rc = dfm.sgemm_watchdog_selftest(timeout_ns=20_000_000)
    assert rc == dfm.STATUS["SGEMM_ERR_WATCHDOG"]
    assert dfm.sgemm_watchdog_status()[0] == 0   # read-and-clear
    run_case(130, 130, 40, "integers", 3)          # device still usable


# The 32 x 32 small-tile kernel on padded, misaligned and multi-chunk k
# layouts (sentinels around C, NaN in the pitch padding of A and B).
@pytest.mark.parametrize("mnk", [(127, 129, 33), (64, 64, 64), (33, 65, 97),
                                 (256, 256, 256), (1, 40, 7), (40, 1, 7)],
                         ids=str)
def test_small_path_layouts(mnk):
    M, N, K = mnk
    for kind in ("uniform", "integers"):
        run_case(M, N, K, kind=kind, seed=M + N + K, path="small")
    run_case(M, N, K, kind="uniform", seed=3, path="small", lda=K + 3,
             ldb=N + 5, ldc=N + 1, offsets=(1, 2, 3))
