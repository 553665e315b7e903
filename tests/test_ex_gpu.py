"""Parity of sgemm_ex (C = alpha * op(A) * op(B) + beta * C) with the CPU
oracle's general form, through the C ABI, on every kernel path.

Operands are stored as the op says (A as K x M for "T", B as N x K for
"T"), uploaded with NaN-poisoned pitch padding and guard bands; C starts
from seeded values (or NaN when beta == 0: it must not be read) inside a
sentinel-filled pitch that must stay untouched. Integer data with
power-of-two scalars stays exact (bit-exact comparison); otherwise the bound
|C - C_oracle| <= 1e-4 * S + 1e-6 with S = |alpha| sum |products| + |beta C0|."""
import numpy as np
import pytest

import matgen
import oracle
from gpu_util import upload, download_c, compare, sample_indices, \
    SENTINEL_BITS

pytestmark = pytest.mark.gpu

OPS = [("N", "N"), ("N", "T"), ("T", "N"), ("T", "T")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_fp32_matrix_gb300 import build
    build.build()


def round4(x):
    return (max(x, 1) + 3) // 4 * 4


def run_ex(op_a, op_b, M, N, K, alpha, beta, kind="uniform", seed=0,
           path="auto", pad=4, check="full", nan_c=None, nan_ab=False):
    import torch
    import dense_fp32_matrix_gb300 as dfm
    gen = matgen.KINDS[kind]
    A = gen(seed, matgen.MATRIX_A, M, K) if M * K else np.zeros((M, K), np.float32)
    B = gen(seed, matgen.MATRIX_B, K, N) if K * N else np.zeros((K, N), np.float32)
    if nan_ab:
        A = np.full_like(A, np.nan)
        B = np.full_like(B, np.nan)
    A_st = np.ascontiguousarray(A if op_a == "N" else A.T)
    B_st = np.ascontiguousarray(B if op_b == "N" else B.T)
    ar, ac = A_st.shape
    br, bc = B_st.shape
    lda, ldb, ldc = round4(ac) + pad, round4(bc) + pad, round4(N) + pad
    C0 = gen(seed, 2, M, N)
    if nan_c is None:
        nan_c = beta == 0.0
    C_in = np.full((M, N), np.nan, np.float32) if nan_c else C0
    bufA, pA = upload(A_st, ar, ac, lda)
    bufB, pB = upload(B_st, br, bc, ldb)
    bufC, pC = upload(C_in, M, N, ldc, fill_bits=SENTINEL_BITS)
    dfm.sgemm_ex(op_a, op_b, M, N, K, alpha, pA, lda, pB, ldb, beta, pC, ldc,
                 path=path)
    torch.cuda.synchronize()
    assert dfm.sgemm_watchdog_status() == (0, 0)
    got = download_c(bufC, M, N, ldc)
    what = "sgemm_ex %s%s %dx%dx%d a=%g b=%g %s %s" % (
        op_a, op_b, M, N, K, alpha, beta, kind, path)
    if check == "full":
        ref, S = oracle.gemm_ex(op_a, op_b, alpha, None if nan_ab else A_st,
                                None if nan_ab else B_st, beta,
                                None if beta == 0.0 else C0, M, N, K)
        return compare(kind, got, ref, S, what)
    # large shapes (alpha = 1, beta = 0): sampled rows of the plain product
    assert alpha == 1.0 and beta == 0.0
    rows, _, _ = sample_indices(M, N)
    ref, S = oracle.gemm_rows(A, B, rows)
    return compare(kind, got[rows], ref, S, what + " rows")


PATHS_2D = ["auto", "tf32x3", "tf32x3_pair", "tiled_tma", "tiled_ldg", "naive",
            "small"]


@pytest.mark.parametrize("path", PATHS_2D)
@pytest.mark.parametrize("ops", OPS, ids="".join)
@pytest.mark.parametrize("mnk", [(300, 260, 100), (129, 388, 68)], ids=str)
def test_ops_on_every_path(ops, path, mnk):
    run_ex(*ops, *mnk, 1.0, 0.0, "integers", seed=sum(mnk), path=path)
    run_ex(*ops, *mnk, 1.0, 0.0, "uniform", seed=sum(mnk), path=path)


@pytest.mark.parametrize("path", ["auto", "tf32x3_pair", "tiled_tma",
                                  "tiled_ldg"])
@pytest.mark.parametrize("ops", OPS, ids="".join)
@pytest.mark.parametrize("ab", [(2.0, 1.0), (-0.5, 0.25), (1.0, -1.0)],
                         ids=str)
def test_scalars_exact_on_integers(ops, ab, path):
    run_ex(*ops, 260, 300, 72, *ab, "integers", seed=7, path=path)


@pytest.mark.parametrize("ops", OPS, ids="".join)
@pytest.mark.parametrize("path", ["auto", "tiled_tma"])
def test_general_scalars(ops, path):
    run_ex(*ops, 520, 392, 200, -1.5, 0.7, "uniform", seed=8, path=path)
    run_ex(*ops, 520, 392, 200, 0.3, 0.0, "normal", seed=9, path=path)


@pytest.mark.parametrize("ops", OPS, ids="".join)
def test_beta_zero_does_not_read_c(ops):
    run_ex(*ops, 200, 136, 40, 1.0, 0.0, "uniform", seed=10, nan_c=True)


@pytest.mark.parametrize("ops", OPS, ids="".join)
def test_alpha_zero_does_not_read_a_or_b(ops):
    run_ex(*ops, 200, 136, 40, 0.0, 0.5, "integers", seed=11, nan_ab=True)
    run_ex(*ops, 200, 136, 40, 0.0, 0.0, "integers", seed=11, nan_ab=True)
    run_ex(*ops, 200, 136, 40, 0.0, 1.0, "integers", seed=11, nan_ab=True)


@pytest.mark.parametrize("ops", OPS, ids="".join)
def test_empty_sum_scales_c(ops):
    run_ex(*ops, 70, 90, 0, 1.0, -2.0, "integers", seed=12)
    run_ex(*ops, 70, 90, 0, 1.0, 0.0, "integers", seed=12)


@pytest.mark.parametrize("ops", OPS, ids="".join)
@pytest.mark.parametrize("mnk", [(1, 4096, 512), (1, 37, 129), (4096, 1, 512),
                                 (129, 1, 37), (1, 1, 300)], ids=str)
def test_vector_shapes(ops, mnk):
    run_ex(*ops, *mnk, 1.0, 0.0, "integers", seed=13)
    run_ex(*ops, *mnk, -0.5, 0.25, "uniform", seed=14)


@pytest.mark.parametrize("ops", OPS, ids="".join)
def test_large_transposed_products(ops):
    run_ex(*ops, 4096, 4096, 4096, 1.0, 0.0, "uniform", seed=15,
           check="sampled")


@pytest.mark.parametrize("ops", OPS, ids="".join)
def test_unaligned_transposed_products(ops):
    run_ex(*ops, 1023, 1025, 257, 1.0, 0.0, "uniform", seed=16, pad=1)
    run_ex(*ops, 1023, 1025, 257, 1.0, 0.0, "integers", seed=16, pad=1)


def test_plain_form_matches_sgemm_bitwise():
    import torch
    import dense_fp32_matrix_gb300 as dfm
    for (M, N, K) in [(4096, 4096, 4096), (300, 260, 100), (1, 512, 64),
                      (4095, 4097, 1023)]:
        A = torch.from_numpy(matgen.uniform(17, 0, M, K)).cuda()
        B = torch.from_numpy(matgen.uniform(17, 1, K, N)).cuda()
        C1 = torch.empty(M, N, device="cuda")
        C2 = torch.full((M, N), float("nan"), device="cuda")
        dfm.sgemm(M, N, K, A, K, B, N, C1, N)
        dfm.sgemm_ex("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C2, N)
        torch.cuda.synchronize()
        assert torch.equal(C1, C2), (M, N, K)


@pytest.mark.parametrize("ops", OPS, ids="".join)
def test_pair_matches_one_sm_kernel_bitwise(ops):
    # Whole-tile schedules (short K) sum the same products in the same k
    # order in both tensor-core kernels, for every operand form.
    import torch
    import dense_fp32_matrix_gb300 as dfm
    M, N, K = 2048, 4096, 128
    outs = []
    for path in ("tf32x3", "tf32x3_pair"):
        A = matgen.normal(18, 0, M, K)
        B = matgen.normal(18, 1, K, N)
        A_st = torch.from_numpy(np.ascontiguousarray(A if ops[0] == "N" else A.T)).cuda()
        B_st = torch.from_numpy(np.ascontiguousarray(B if ops[1] == "N" else B.T)).cuda()
        C = torch.empty(M, N, device="cuda")
        dfm.sgemm_ex(ops[0], ops[1], M, N, K, 1.0, A_st, A_st.shape[1], B_st,
                     B_st.shape[1], 0.0, C, N, path=path)
        outs.append(C)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


# c = A^T b with A stored K x M and dense c, b: the M == 1 kernel streams A
# as stored (c^T = b^T A), no transposed copy. Both forms of b, alpha/beta,
# ragged sizes, a row pitch with padding (lda > M), and an unaligned pitch
# (the plain-load row kernel).
@pytest.mark.parametrize("op_b", ["N", "T"])
@pytest.mark.parametrize("M,K,lda_pad", [(4096, 4096, 0), (1000, 3000, 4),
                                         (37, 5000, 3), (3001, 17, 0)],
                         ids=str)
@pytest.mark.parametrize("kind,alpha,beta", [("integers", 0.5, 2.0),
                                             ("uniform", 1.0, 0.0)])
def test_transposed_a_times_vector(op_b, M, K, lda_pad, kind, alpha, beta):
    import torch
    import dense_fp32_matrix_gb300 as dfm
    gen = matgen.KINDS[kind]
    A = gen(5, matgen.MATRIX_A, M, K)
    b = gen(5, matgen.MATRIX_B, K, 1)
    C0 = gen(5, 2, M, 1)
    A_st = np.ascontiguousarray(A.T)                    # K x M
    lda = M + lda_pad
    assert dfm.sgemm_plan_ex("T", op_b, M, 1, K, lda, K if op_b == "T" else 1,
                             1, 0x7f0000000000, 0x7f0010000000,
                             0x7f0020000000) == "gemv_row"
    dA = torch.full((K, lda), float("nan"), device="cuda")
    dA[:, :M] = torch.from_numpy(A_st)
    db = torch.from_numpy(np.ascontiguousarray(b.ravel())).cuda()
    dC = torch.from_numpy(np.ascontiguousarray(C0.ravel())).cuda()
    dfm.sgemm_ex("T", op_b, M, 1, K, alpha, dA, lda, db,
                 K if op_b == "T" else 1, beta, dC, 1)
    torch.cuda.synchronize()
    assert dfm.sgemm_watchdog_status() == (0, 0)
    ref, S = oracle.gemm_ex("T", op_b, alpha, A_st,
                            b.reshape(1, K) if op_b == "T" else b, beta, C0,
                            M, 1, K)
    compare(kind, dC.cpu().numpy().reshape(M, 1), ref, S,
            "A^T b %dx%d %s" % (M, K, op_b))
