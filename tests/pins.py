"""Pins for the CPU oracle: checks that do not go through the oracle itself.

Each pin takes ``gemm(A, B) -> C`` (dense fp32 numpy inputs, fp64 output)
and raises AssertionError when the function disagrees with what the pages or
mathematics fix. The pins are chosen so that the plausible slips in a matrix
product (a dropped term, a transposed operand, a wrong sign, a shifted index,
a misused leading dimension) each fail at least one of them;
tests/test_oracle_pins.py checks that claim against planted mistakes.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

import matgen


def _rng(seed):
    return np.random.default_rng(seed)


def pin_identity(gemm):
    """A * I = A and I * B = B exactly: each output is one product plus zeros
    (definition of the product, "CUDA 算子优化：GEMM", section 矩阵乘法)."""
    A = matgen.uniform(11, 0, 37, 29)
    C = gemm(A, np.eye(29, dtype=np.float32))
    assert np.array_equal(C, A.astype(np.float64)), "A*I != A"
    B = matgen.uniform(11, 1, 23, 41)
    C = gemm(np.eye(23, dtype=np.float32), B)
    assert np.array_equal(C, B.astype(np.float64)), "I*B != B"


def pin_all_ones(gemm):
    """All-ones operands give C_ij = K exactly, for ragged and tiny shapes."""
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (17, 9, 33), (5, 4, 129)]:
        C = gemm(np.ones((M, K), np.float32), np.ones((K, N), np.float32))
        assert C.shape == (M, N)
        assert np.all(C == K), "all-ones product must equal K"


def pin_rank1(gemm):
    """K = 1: C = a b^T, each entry one exact fp64 product (the rank-1 update
    of the outer-product view, hotelren.com section 1.3)."""
    a = matgen.uniform(12, 0, 19, 1)
    b = matgen.uniform(12, 1, 1, 23)
    C = gemm(a, b)
    ref = np.multiply.outer(a[:, 0].astype(np.float64), b[0].astype(np.float64))
    assert np.array_equal(C, ref), "rank-1 product"


def pin_closed_forms(gemm):
    """Index-revealing closed forms.

    A_ik = k, B = ones      -> C_ij = K(K-1)/2   (catches a transposed A)
    A = ones, B_kj = k      -> C_ij = K(K-1)/2   (catches a transposed B)
    A_ik = i+1, B_kj = j+1  -> C_ij = K(i+1)(j+1)
    A_ik = 1, B_kj = (-1)^k -> C_ij = 1 if K odd else 0   (catches a sign slip)
    """
    M, N, K = 13, 11, 17
    A = np.tile(np.arange(K, dtype=np.float32), (M, 1))
    C = gemm(A, np.ones((K, N), np.float32))
    assert np.all(C == K * (K - 1) / 2)
    B = np.tile(np.arange(K, dtype=np.float32)[:, None], (1, N))
    C = gemm(np.ones((M, K), np.float32), B)
    assert np.all(C == K * (K - 1) / 2)
    A = np.tile(np.arange(1, M + 1, dtype=np.float32)[:, None], (1, K))
    B = np.tile(np.arange(1, N + 1, dtype=np.float32), (K, 1))
    C = gemm(A, B)
    i = np.arange(1, M + 1)[:, None]
    j = np.arange(1, N + 1)[None, :]
    assert np.array_equal(C, (K * i * j).astype(np.float64))
    B = np.tile(((-1.0) ** np.arange(K)).astype(np.float32)[:, None], (1, N))
    C = gemm(np.ones((M, K), np.float32), B)
    assert np.all(C == (1.0 if K % 2 else 0.0))


def pin_permutation(gemm):
    """A permutation matrix P: P * B reorders the rows of B exactly."""
    perm = _rng(3).permutation(15)
    P = np.zeros((15, 15), np.float32)
    P[np.arange(15), perm] = 1.0
    B = matgen.uniform(13, 1, 15, 21)
    assert np.array_equal(gemm(P, B), B[perm].astype(np.float64))


def pin_brute_force_exact(gemm, sizes=(1, 2, 3, 4, 5, 7, 8, 9, 16, 17)):
    """Tiny integer shapes against exact Python-integer sums.

    For integer inputs in [-4, 4] every partial sum is an integer far below
    2**53, so the fp64 result must equal the exact sum bit for bit.
    """
    seed = 0
    for M in sizes[::3]:
        for N in sizes[1::3]:
            for K in sizes:
                seed += 1
                A = matgen.integers(seed, 0, M, K)
                B = matgen.integers(seed, 1, K, N)
                Ai = A.astype(np.int64).tolist()
                Bi = B.astype(np.int64).tolist()
                exact = [[sum(Ai[i][k] * Bi[k][j] for k in range(K))
                          for j in range(N)] for i in range(M)]
                C = gemm(A, B)
                assert np.array_equal(C, np.array(exact, dtype=np.float64)), \
                    (M, N, K)


def pin_exact_rational(gemm):
    """Uniform fp32 inputs: compare with the exact rational sum.

    The fp64 sum of K exact products in any order is within K * 2**-53 * S
    of the exact value (S = sum |A_ik B_kj|); the oracle must be inside it.
    """
    for (M, N, K, seed) in [(4, 5, 9, 21), (3, 3, 31, 22), (2, 6, 64, 23)]:
        A = matgen.uniform(seed, 0, M, K)
        B = matgen.uniform(seed, 1, K, N)
        C = gemm(A, B)
        for i in range(M):
            for j in range(N):
                terms = [Fraction(float(A[i, k])) * Fraction(float(B[k, j]))
                         for k in range(K)]
                exact = sum(terms, Fraction(0))
                S = float(sum(abs(t) for t in terms))
                err = abs(Fraction(float(C[i, j])) - exact)
                assert err <= Fraction(K * S) / 2 ** 53, (i, j)


def pin_library(gemm):
    """Cross-check with numpy's fp64 matrix product (an independent summation
    order) within the fp64 rounding bound K * 2**-52 * S."""
    M, N, K = 33, 47, 129
    A = matgen.normal(31, 0, M, K)
    B = matgen.normal(31, 1, K, N)
    A64, B64 = A.astype(np.float64), B.astype(np.float64)
    ref = A64 @ B64
    S = np.abs(A64) @ np.abs(B64)
    C = gemm(A, B)
    assert np.all(np.abs(C - ref) <= K * 2.0 ** -52 * S + 1e-300)


def pin_zero_padding(gemm):
    """Zero padding leaves C unchanged. Shapes from the boundary-handling
    example of "GEMM from naive to tiled", section 七: M, N, K = 300, 200, 20
    padded to 384 x 256 x 24 (zero rows/columns contribute 0 * b = 0)."""
    M, N, K = 300, 200, 20
    A = matgen.uniform(41, 0, M, K)
    B = matgen.uniform(41, 1, K, N)
    Ap = np.zeros((384, 24), np.float32)
    Bp = np.zeros((24, 256), np.float32)
    Ap[:M, :K] = A
    Bp[:K, :N] = B
    C = gemm(A, B)
    Cp = gemm(Ap, Bp)
    assert np.array_equal(Cp[:M, :N], C)
    assert np.all(Cp[M:, :] == 0) and np.all(Cp[:, N:] == 0)


ALL_PINS = [pin_identity, pin_all_ones, pin_rank1, pin_closed_forms,
            pin_permutation, pin_brute_force_exact, pin_exact_rational,
            pin_library, pin_zero_padding]
