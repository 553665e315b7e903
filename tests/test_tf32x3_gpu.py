"""Parity of the 3xTF32 tensor-core path with the CPU oracle (C ABI).

Same bar as every other path: bit-exact on integer data (the split leaves
lo = 0 and TF32 products of small integers are exact), |C - C_oracle| <=
1e-4 * S + 1e-6 otherwise. The path needs 16-byte row strides (K and N
multiples of 4 for dense matrices)."""
import itertools

import numpy as np
import pytest

import matgen
import oracle
from matgen.workloads import WORKLOADS
from gpu_util import compare, run_case

pytestmark = pytest.mark.gpu

PATH = "tf32x3"          # one block per 128 x 128 tile
PAIR = "tf32x3_pair"     # 2-SM clusters, 256 x 256 tiles


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_fp32_matrix_gb300 import build
    build.build()


ALIGNED = [w for w in WORKLOADS if w["K"] % 4 == 0 and w["N"] % 4 == 0]


@pytest.mark.parametrize("path", [PATH, PAIR])
@pytest.mark.parametrize("w", ALIGNED, ids=lambda w: w["name"])
def test_workload(w, path):
    worst = run_case(w["M"], w["N"], w["K"], w["kind"], w["seed"], path=path)
    if w["kind"] != "integers":
        # the split's extra error is ~3 * 2^-20 of each |product|
        assert worst < 0.25


@pytest.mark.parametrize("mnk", [(300, 200, 20), (260, 132, 36), (129, 260, 68),
                                 (1000, 1000, 1000), (128, 128, 32),
                                 (384, 256, 24), (1, 4096, 256), (4096, 4, 64)],
                         ids=str)
@pytest.mark.parametrize("kind", ["uniform", "integers", "normal"])
@pytest.mark.parametrize("path", [PATH, PAIR])
def test_multi_tile(mnk, kind, path):
    run_case(*mnk, kind=kind, seed=sum(mnk), path=path)


@pytest.mark.parametrize("path", [PATH, PAIR])
def test_tiny_aligned_shapes_bit_exact(path):
    for M, N, K in itertools.product((1, 2, 3, 5, 8, 17, 33, 129),
                                     (4, 8, 12, 36, 132), (4, 8, 12, 36, 68)):
        run_case(M, N, K, kind="integers", seed=M * 7 + N * 3 + K, path=path,
                 check="full")


@pytest.mark.parametrize("path", [PATH, PAIR])
def test_pitch_padding_never_read_or_written(path):
    run_case(300, 200, 64, "uniform", 9, lda=72, ldb=204, ldc=260, path=path)
    run_case(260, 132, 36, "integers", 9, lda=40, ldb=136, ldc=133, path=path)


@pytest.mark.parametrize("path", [PATH, PAIR])
def test_misaligned_operands_are_repacked(path):
    # Row strides or bases that are not 16-byte aligned are copied with an
    # aligned stride before the tensor maps are made (same results bar).
    run_case(64, 64, 33, "integers", 3, path=path, check="full")
    run_case(300, 260, 101, "uniform", 4, lda=103, ldb=263, ldc=261, path=path)
    run_case(257, 130, 77, "integers", 5, path=path, offsets=(1, 3, 2))
    run_case(1000, 1030, 513, "uniform", 6, path="auto", offsets=(1, 1, 1))


def test_nan_and_inf_propagate():
    import torch
    import dense_fp32_matrix_gb300 as dfm
    A = torch.from_numpy(matgen.uniform(1, 0, 256, 256)).cuda()
    B = torch.from_numpy(matgen.uniform(1, 1, 256, 256)).cuda()
    A[7, 100] = float("nan")
    B[30, 200] = float("nan")
    C = dfm.matmul(A, B, path=PATH)
    torch.cuda.synchronize()
    nan = torch.isnan(C).cpu().numpy()
    assert nan[7].all() and nan[:, 200].all()
    nan[7] = False
    nan[:, 200] = False
    assert not nan.any()
    # An infinite input makes its row non-finite. (On this path it comes out
    # as NaN, not inf: the compensation term A_hi * B_lo multiplies the
    # infinity by an exactly-zero residual.)
    A = torch.ones(128, 128, device="cuda")
    A[3, 5] = float("inf")
    C = dfm.matmul(A, torch.ones(128, 128, device="cuda"), path=PATH)
    torch.cuda.synchronize()
    assert not torch.isfinite(C[3]).any()
    assert torch.isfinite(C[:3]).all() and torch.isfinite(C[4:]).all()


def test_auto_dispatch_picks_the_tensor_path_for_aligned_operands():
    import torch
    import dense_fp32_matrix_gb300 as dfm
    A = torch.from_numpy(matgen.integers(3, 0, 640, 388)).cuda()
    B = torch.from_numpy(matgen.integers(3, 1, 388, 260)).cuda()
    assert dfm.sgemm_plan(640, 260, 388, 388, 260, 260, A.data_ptr(),
                          B.data_ptr(), 0x7f0020000000) == PATH
    run_case(640, 260, 388, "integers", 3, path="auto")
    assert dfm.sgemm_plan(2048, 2048, 260, 260, 2048, 2048, A.data_ptr(),
                          B.data_ptr(), 0x7f0020000000) == PAIR
    run_case(2048, 2048, 260, "integers", 3, path="auto")


@pytest.mark.parametrize("path", [PATH, PAIR])
def test_deterministic(path):
    import torch
    import dense_fp32_matrix_gb300 as dfm
    A = torch.from_numpy(matgen.uniform(2, 0, 1000, 780)).cuda()
    B = torch.from_numpy(matgen.uniform(2, 1, 780, 996)).cuda()
    C1 = dfm.matmul(A, B, path=path)
    C2 = dfm.matmul(A, B, path=path)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)


# Shapes that drive each branch of the pair kernel's persistent schedule on
# a 152-SM part (76 clusters): whole waves plus a stream-K tail, a tail
# widened by one wave (one tile over a wave), every tile split by k-slices
# (fewer tiles than clusters), whole tiles only (short K), and ragged edges
# in M, N and K inside split tiles.
PAIR_SCHEDULES = [
    (4096, 4096, 4096),    # 228 whole + 28 split
    (1792, 2816, 1024),    # 77 tiles: the split part widened to 77
    (1000, 1000, 1000),    # 16 tiles over 64 clusters
    (2048, 2048, 2048),    # 64 tiles over 76 clusters
    (4096, 4096, 64),      # 2 k-slices: whole tiles, round robin
    (2300, 2900, 1900),    # ragged M, N, K; split tiles at the edges
    (20000, 260, 516),     # tall and thin
]


@pytest.mark.parametrize("mnk", PAIR_SCHEDULES, ids=str)
@pytest.mark.parametrize("kind", ["uniform", "integers"])
def test_pair_schedules(mnk, kind):
    run_case(*mnk, kind=kind, seed=sum(mnk) % 1000, path=PAIR)


def test_pair_split_tiles_deterministic():
    import torch
    import dense_fp32_matrix_gb300 as dfm
    A = torch.from_numpy(matgen.normal(5, 0, 2300, 1900)).cuda()
    B = torch.from_numpy(matgen.normal(5, 1, 1900, 2900)).cuda()
    outs = [dfm.matmul(A, B, path=PAIR) for _ in range(3)]
    torch.cuda.synchronize()
    assert all(torch.equal(outs[0], o) for o in outs[1:])


def test_concurrent_streams_do_not_share_partials():
    # Two unordered streams run split-tile products at the same time; each
    # stream has its own stream-K workspace, so both match the serial result.
    import torch
    import dense_fp32_matrix_gb300 as dfm
    A = torch.from_numpy(matgen.uniform(6, 0, 2300, 1900)).cuda()
    B = torch.from_numpy(matgen.uniform(6, 1, 1900, 2900)).cuda()
    A2 = torch.from_numpy(matgen.uniform(7, 0, 2300, 1900)).cuda()
    ref = dfm.matmul(A, B, path=PAIR)
    ref2 = dfm.matmul(A2, B, path=PAIR)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(4):
        C1 = torch.empty_like(ref)
        C2 = torch.empty_like(ref)
        with torch.cuda.stream(s1):
            dfm.matmul(A, B, out=C1, path=PAIR)
        with torch.cuda.stream(s2):
            dfm.matmul(A2, B, out=C2, path=PAIR)
        outs.append((C1, C2))
    torch.cuda.synchronize()
    assert dfm.sgemm_watchdog_status() == (0, 0)
    for C1, C2 in outs:
        assert torch.equal(C1, ref)
        assert torch.equal(C2, ref2)


# The pair kernel leaves the landed A in place as its TF32 high part (the
# MMA reads an fp32 operand as TF32 by ignoring the 13 low mantissa bits);
# the 1-SM kernel writes the masked high part. On schedules of whole tiles
# both sum the same three products in the same k order, so the results must
# agree bit for bit. Short K keeps the pair schedule to whole tiles on any
# cluster count; 1024 x 4864 is one full wave of 76 pair tiles on a
# 152-SM GB300.
@pytest.mark.parametrize("mnk", [(4096, 4096, 64), (2048, 4096, 128),
                                 (1024, 4864, 1000)], ids=str)
@pytest.mark.parametrize("kind", ["uniform", "normal"])
def test_pair_matches_masked_high_part_bitwise(mnk, kind):
    import torch
    import dense_fp32_matrix_gb300 as dfm
    M, N, K = mnk
    if K > 128 and torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("one full wave of pair tiles needs 152 SMs")
    A = torch.from_numpy(matgen.KINDS[kind](11, 0, M, K)).cuda()
    B = torch.from_numpy(matgen.KINDS[kind](11, 1, K, N)).cuda()
    C1 = dfm.matmul(A, B, path=PATH)
    C2 = dfm.matmul(A, B, path=PAIR)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)


# Schedules with whole tiles after the stream-K shares (2300 x 2900 x 1900:
# 108 tiles, 76 whole + 32 split on 76 clusters) sum a split tile's pieces
# as soon as the last one is in and write C straight from registers: alpha,
# beta, and rows that are not 16-byte aligned (pad 1) all go through it.
@pytest.mark.parametrize("pad", [4, 1])
@pytest.mark.parametrize("ops", [("N", "N"), ("T", "T")], ids="".join)
@pytest.mark.parametrize("kind,alpha,beta", [("integers", 0.5, 2.0),
                                             ("uniform", 0.75, -1.5),
                                             ("uniform", 1.0, 0.0)])
def test_pair_early_fixup_epilogue(pad, ops, kind, alpha, beta):
    from test_ex_gpu import run_ex
    run_ex(*ops, 2300, 2900, 1900, alpha, beta, kind=kind, seed=7, path=PAIR,
           pad=pad)


# C with rows that do not end on a 16-byte boundary (N % 4 != 0) inside a
# 16-byte-aligned pitch: a bulk tensor store writes whole 16-byte chunks, so
# these must take the staged row stores; the pitch padding stays untouched
# (whole tiles, split tiles, every tile split).
@pytest.mark.parametrize("mnk,ldc", [((1893, 1777, 426), 1780),
                                     ((2300, 2901, 1900), 2904),
                                     ((1000, 1001, 1000), 1004),
                                     ((300, 203, 64), 208)], ids=str)
def test_pair_never_writes_past_row_end(mnk, ldc):
    run_case(*mnk, kind="integers", seed=5, ldc=ldc, path=PAIR)


# Few tiles: the single-block kernel splits k over the idle SMs and a
# second kernel adds the pieces in order (alpha, beta, ragged edges,
# transposed forms and batches all go through the reduce kernel).
@pytest.mark.parametrize("ops", [("N", "N"), ("N", "T"), ("T", "N"), ("T", "T")],
                         ids="".join)
@pytest.mark.parametrize("kind,alpha,beta", [("integers", 0.5, 2.0),
                                             ("uniform", -1.25, 0.5),
                                             ("uniform", 1.0, 0.0)])
def test_split_k_single_blocks(ops, kind, alpha, beta):
    from test_ex_gpu import run_ex
    run_ex(*ops, 700, 300, 900, alpha, beta, kind=kind, seed=3, path=PATH)
    run_ex(*ops, 129, 1000, 4000, alpha, beta, kind=kind, seed=4, path=PATH,
           pad=1)


@pytest.mark.parametrize("side", [False, True])
def test_split_k_batches(side):
    from test_batched_gpu import run_batch
    run_batch(("N", "N"), 200, 300, 640, 3, alpha=0.5, beta=2.0,
              kind="integers", seed=8, path=PATH, side_by_side=side)
    run_batch(("T", "N"), 257, 129, 1000, 2, kind="uniform", seed=9,
              path=PATH, shared_b=True, side_by_side=side)


def test_split_k_matches_unsplit_bitwise_on_integers():
    # integer data: every split and the single pass are exact, so equal
    import torch
    import dense_fp32_matrix_gb300 as dfm
    A_h = matgen.integers(12, 0, 512, 2048)
    B_h = matgen.integers(12, 1, 2048, 384)
    A = torch.from_numpy(A_h).cuda()
    B = torch.from_numpy(B_h).cuda()
    C = dfm.matmul(A, B, path=PATH)       # 12 tiles: split k
    ref, S = oracle.gemm(A_h, B_h)
    torch.cuda.synchronize()
    compare("integers", C.cpu().numpy(), ref, S, "split k")
    # and another split of the same products (the pair kernel's stream-K
    # schedule): exact sums, so the same bits
    C1 = dfm.matmul(A, B, path=PAIR)
    torch.cuda.synchronize()
    assert torch.equal(C, C1)
