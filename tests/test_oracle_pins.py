"""The CPU oracle against checks that do not come from the oracle itself."""
import numpy as np
import pytest

import matgen
import oracle
from pins import ALL_PINS


def oracle_outer(A, B):
    return oracle.gemm(A, B, order="outer", with_abs=False)[0]


def oracle_inner(A, B):
    return oracle.gemm(A, B, order="inner", with_abs=False)[0]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
@pytest.mark.parametrize("fn", [oracle_outer, oracle_inner],
                         ids=["outer", "inner"])
def test_oracle_passes_pin(pin, fn):
    pin(fn)


# -- planted mistakes: each must be caught by at least one pin --------------

def _mut_drop_last(A, B):
    return oracle_outer(np.ascontiguousarray(A[:, :-1]),
                        np.ascontiguousarray(B[:-1]))


def _mut_drop_first(A, B):
    return oracle_outer(np.ascontiguousarray(A[:, 1:]),
                        np.ascontiguousarray(B[1:]))


def _mut_transposed_a(A, B):
    # reads A[k * M + i] instead of A[i * K + k]
    M, K = A.shape
    return oracle_outer(np.ascontiguousarray(A.reshape(K, M).T), B)


def _mut_transposed_b(A, B):
    K, N = B.shape
    return oracle_outer(A, np.ascontiguousarray(B.reshape(N, K).T))


def _mut_wrong_sign(A, B):
    B2 = B.copy()
    B2[-1] = -B2[-1]
    return oracle_outer(A, B2)


def _mut_shifted_column(A, B):
    return oracle_outer(A, np.ascontiguousarray(np.roll(B, -1, axis=1)))


def _mut_fp32_accumulation(A, B):
    M, K = A.shape
    N = B.shape[1]
    C = np.zeros((M, N), np.float32)
    for k in range(K):
        C = (C + np.multiply.outer(A[:, k], B[k]).astype(np.float32)).astype(
            np.float32)
    return C.astype(np.float64)


MUTANTS = [_mut_drop_last, _mut_drop_first, _mut_transposed_a,
           _mut_transposed_b, _mut_wrong_sign, _mut_shifted_column,
           _mut_fp32_accumulation]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_pins_catch_planted_mistake(mutant):
    caught = []
    for pin in ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, "no pin caught %s" % mutant.__name__


# -- leading dimensions, subsets, degenerate sizes, argument errors ---------

def test_pitch_padding_is_never_read():
    M, N, K = 19, 23, 29
    A = matgen.make("uniform", 5, 0, M, K, ld=K + 7)   # NaN in the padding
    B = matgen.make("uniform", 5, 1, K, N, ld=N + 3)
    C, S = oracle.gemm(A, B, M=M, N=N, K=K, lda=K + 7, ldb=N + 3)
    Cd, Sd = oracle.gemm(np.ascontiguousarray(A[:, :K]),
                         np.ascontiguousarray(B[:, :N]))
    assert np.isfinite(C).all()
    assert np.array_equal(C, Cd) and np.array_equal(S, Sd)


def test_rows_and_entries_match_full():
    M, N, K = 41, 37, 53
    A = matgen.uniform(6, 0, M, K)
    B = matgen.uniform(6, 1, K, N)
    C, S = oracle.gemm(A, B)
    rows = [0, 7, 40]
    Cr, Sr = oracle.gemm_rows(A, B, rows)
    assert np.array_equal(Cr, C[rows]) and np.array_equal(Sr, S[rows])
    ii = np.array([0, 40, 13, 5])
    jj = np.array([36, 0, 13, 22])
    c, s = oracle.gemm_entries(A, B, ii, jj)
    assert np.array_equal(c, C[ii, jj]) and np.array_equal(s, S[ii, jj])


def test_abs_sum_scale():
    A = np.array([[1, -2]], np.float32)
    B = np.array([[3], [4]], np.float32)
    C, S = oracle.gemm(A, B)
    assert C[0, 0] == -5.0 and S[0, 0] == 11.0


def test_degenerate_sizes():
    C, S = oracle.gemm(np.zeros((4, 0), np.float32), np.zeros((0, 5), np.float32),
                       M=4, N=5, K=0, lda=1, ldb=5)
    assert C.shape == (4, 5) and np.all(C == 0) and np.all(S == 0)
    C, _ = oracle.gemm(np.zeros((0, 3), np.float32), np.ones((3, 5), np.float32),
                       M=0, N=5, K=3, lda=3, ldb=5)
    assert C.shape == (0, 5)
    C, _ = oracle.gemm(np.ones((2, 3), np.float32), np.zeros((3, 0), np.float32),
                       M=2, N=0, K=3, lda=3, ldb=1)
    assert C.shape == (2, 0)


def test_invalid_arguments_rejected():
    A = np.ones((4, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.gemm(A, A, M=4, N=4, K=4, lda=3, ldb=4)
    with pytest.raises(ValueError):
        oracle.gemm(A, A, M=4, N=4, K=4, lda=4, ldb=2)
    with pytest.raises(ValueError):
        oracle.gemm_rows(A, A, [4])


def test_integer_inputs_fp32_rounding_is_exact():
    # |A_ik B_kj| <= 16 and |C| <= 16 K < 2**24 for K up to 11008, so the fp32
    # rounding of the fp64 sum is the exact integer.
    M, N, K = 8, 9, 11008
    A = matgen.integers(9, 0, M, K)
    B = matgen.integers(9, 1, K, N)
    C, _ = oracle.gemm(A, B)
    assert np.all(np.abs(C) <= 16 * K)
    assert np.array_equal(oracle.round_fp32(C).astype(np.float64), C)


def test_threads_reported():
    assert oracle.num_threads() >= 1


# -- the inner-product and outer-product formulations agree ------------------
# hotelren.com, section 1.3: reordering the loops into rank-1 updates does
# not change the mathematical result. Both orders form each exact fp64
# product and add them per output in ascending k, so on float data (not just
# integers) the two results and the two absolute sums agree bit for bit.

@pytest.mark.parametrize("kind", ["uniform", "normal"])
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (7, 5, 3), (33, 17, 65),
                                   (64, 96, 300), (129, 31, 1023)])
def test_inner_equals_outer_bitwise_on_floats(kind, M, N, K):
    A = matgen.KINDS[kind](70 + K, matgen.MATRIX_A, M, K)
    B = matgen.KINDS[kind](70 + K, matgen.MATRIX_B, K, N)
    ci, si = oracle.gemm(A, B, order="inner")
    co, so = oracle.gemm(A, B, order="outer")
    assert np.array_equal(ci.view(np.uint64), co.view(np.uint64))
    assert np.array_equal(si.view(np.uint64), so.view(np.uint64))
    # and the row / entry subsets used for large shapes are the same sums
    rows = np.array([0, M - 1], dtype=np.int64)
    cr, sr = oracle.gemm_rows(A, B, rows)
    assert np.array_equal(cr, co[rows]) and np.array_equal(sr, so[rows])
    ii = np.array([0, M - 1, M // 2], dtype=np.int64)
    jj = np.array([N - 1, 0, N // 2], dtype=np.int64)
    ce, se = oracle.gemm_entries(A, B, ii, jj)
    assert np.array_equal(ce, co[ii, jj]) and np.array_equal(se, so[ii, jj])
