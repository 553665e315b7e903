"""Pins of the oracle's general form alpha * op(A) * op(B) + beta * C0.

Each pin ties it to something other than itself: the already-pinned plain
product (oracle.gemm) through transposes made by numpy, the identity
(A B)^T = B^T A^T, exact scalings by powers of two, the BLAS rules for
alpha == 0 / beta == 0 (unread operands may hold NaN), and exact integer
sums. test_ex_pins_catch_planted_mistakes plants plausible mistakes in
wrappers of the oracle and checks that each one fails a pin."""
import numpy as np
import pytest

import matgen
import oracle

SHAPES = [(1, 1, 1), (3, 5, 7), (17, 9, 33), (64, 48, 40), (5, 1, 8)]


def _ints(seed, mid, r, c):
    return matgen.integers(seed, mid, r, c)


def stored(X, op):
    """The array to pass for op(X) = X when op == "N", else X^T stored."""
    return np.ascontiguousarray(X if op == "N" else X.T)


def pin_transposes(ex):
    # op(A) op(B) with A, B stored transposed equals the plain product
    for (M, N, K) in SHAPES:
        A = matgen.uniform(M + N, 0, M, K)
        B = matgen.uniform(M + N, 1, K, N)
        ref, S = oracle.gemm(A, B)
        for oa in "NT":
            for ob in "NT":
                C, S2 = ex(oa, ob, 1.0, stored(A, oa), stored(B, ob), 0.0,
                           None, M, N, K)
                assert np.array_equal(C, ref), (oa, ob, M, N, K)
                assert np.array_equal(S2, S)


def pin_transpose_identity(ex):
    # (A B)^T = B^T A^T: with B and A passed "T", C' = op(B) op(A) is the
    # transposed product, element by element the same exact products.
    for (M, N, K) in SHAPES:
        A = _ints(7, 0, M, K)
        B = _ints(7, 1, K, N)
        ref, _ = oracle.gemm(A, B)
        C, _ = ex("T", "T", 1.0, B, A, 0.0, None, N, M, K)
        assert np.array_equal(C, ref.T)


def pin_scalars(ex):
    M, N, K = 12, 10, 9
    A = _ints(3, 0, M, K)
    B = _ints(3, 1, K, N)
    C0 = _ints(3, 2, M, N)
    AB = A.astype(np.float64) @ B.astype(np.float64)     # exact integers
    C, _ = ex("N", "N", 2.0, A, B, 0.0, None, M, N, K)
    assert np.array_equal(C, 2.0 * AB)
    C, _ = ex("N", "N", 1.0, A, B, 1.0, C0, M, N, K)
    assert np.array_equal(C, AB + C0)
    C, _ = ex("N", "N", -0.5, A, B, 0.25, C0, M, N, K)
    assert np.array_equal(C, -0.5 * AB + 0.25 * C0.astype(np.float64))
    # beta == 0: C0 is not read (NaN in it must not appear)
    nan = np.full((M, N), np.nan, np.float32)
    C, _ = ex("N", "N", 1.0, A, B, 0.0, nan, M, N, K)
    assert np.array_equal(C, AB)
    # alpha == 0: A and B are not read
    nanA = np.full((M, K), np.nan, np.float32)
    nanB = np.full((K, N), np.nan, np.float32)
    C, S = ex("N", "N", 0.0, nanA, nanB, 3.0, C0, M, N, K)
    assert np.array_equal(C, 3.0 * C0.astype(np.float64))
    assert np.array_equal(S, np.abs(3.0 * C0.astype(np.float64)))
    # K == 0: C = beta * C0
    C, _ = ex("T", "N", 5.0, None, None, -1.0, C0, M, N, 0)
    assert np.array_equal(C, -C0.astype(np.float64))


def pin_scale(ex):
    # S = |alpha| sum |products| + |beta C0|
    M, N, K = 6, 7, 5
    A = _ints(9, 0, M, K)
    B = _ints(9, 1, K, N)
    C0 = _ints(9, 2, M, N)
    _, S = ex("N", "N", -2.0, A, B, -0.5, C0, M, N, K)
    mag = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
    assert np.array_equal(S, 2.0 * mag + 0.5 * np.abs(C0.astype(np.float64)))


ALL = [pin_transposes, pin_transpose_identity, pin_scalars, pin_scale]


@pytest.mark.parametrize("pin", ALL, ids=lambda f: f.__name__)
def test_oracle_ex_pin(pin):
    pin(oracle.gemm_ex)


def test_ex_rejects_bad_arguments():
    A = np.zeros((3, 4), np.float32)
    B = np.zeros((4, 5), np.float32)
    with pytest.raises(ValueError):          # op(A) needs ld >= M = 6
        oracle.gemm_ex("T", "N", 1.0, A, B, 0.0, None, 6, 5, 3, lda=4)
    with pytest.raises(ValueError):          # beta != 0 without C0
        oracle.gemm_ex("N", "N", 1.0, A, B, 1.0, None, 3, 5, 4)
    with pytest.raises(KeyError):
        oracle.gemm_ex("C", "N", 1.0, A, B, 0.0, None, 3, 5, 4)


def _mutants():
    ex = oracle.gemm_ex

    def swapped_a(oa, ob, al, A, B, be, C0, M, N, K, **kw):
        # reads A as if it were never transposed
        if oa == "T" and A is not None:
            A = np.ascontiguousarray(A.T.reshape(A.shape))
        return ex(oa, ob, al, A, B, be, C0, M, N, K, **kw)

    def swapped_b(oa, ob, al, A, B, be, C0, M, N, K, **kw):
        if ob == "T" and B is not None:
            B = np.ascontiguousarray(B.T.reshape(B.shape))
        return ex(oa, ob, al, A, B, be, C0, M, N, K, **kw)

    def beta_ignored(oa, ob, al, A, B, be, C0, M, N, K, **kw):
        return ex(oa, ob, al, A, B, 0.0, None, M, N, K, **kw)

    def alpha_on_c0(oa, ob, al, A, B, be, C0, M, N, K, **kw):
        C, S = ex(oa, ob, al, A, B, be * al if al != 0 else be, C0, M, N, K,
                  **kw)
        return C, S

    def reads_c0_when_beta_zero(oa, ob, al, A, B, be, C0, M, N, K, **kw):
        if be == 0.0 and C0 is not None:
            C, S = ex(oa, ob, al, A, B, 1e-300, C0, M, N, K, **kw)
            return C + 0.0 * np.asarray(C0, np.float64), S
        return ex(oa, ob, al, A, B, be, C0, M, N, K, **kw)

    def scale_without_alpha(oa, ob, al, A, B, be, C0, M, N, K, **kw):
        C, S = ex(oa, ob, al, A, B, be, C0, M, N, K, **kw)
        if al != 0 and abs(al) != 1:
            S = S - (abs(al) - 1) * ex(oa, ob, 1.0, A, B, 0.0, None, M, N,
                                       K, **kw)[1]
        return C, S
    return [swapped_a, swapped_b, beta_ignored, alpha_on_c0,
            reads_c0_when_beta_zero, scale_without_alpha]


@pytest.mark.parametrize("mutant", _mutants(), ids=lambda f: f.__name__)
def test_ex_pins_catch_planted_mistakes(mutant):
    caught = 0
    for pin in ALL:
        try:
            with np.errstate(all="ignore"):
                pin(mutant)
        except (AssertionError, ValueError):
            caught += 1
    assert caught >= 1, mutant.__name__
