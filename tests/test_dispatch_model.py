"""The library's path choice (sgemm_plan_ex, host-only) against a plain
statement of the dispatch rules, on seeded random arguments (no GPU).

The rules, in order:
  * nothing to compute (M or N = 0, K = 0): no kernel;
  * M == 1: the row-vector kernel, or the column kernel when B is stored
    transposed (c = a Bᵀ are B's rows times a);
  * N == 1: the column kernel, or the row kernel for c = Aᵀ b with A stored
    transposed and c, b contiguous (cᵀ = bᵀ A);
  * at most 2^23 multiply-adds (and M within the kernel's grid): the
    small-tile kernel, in either math mode;
  * in the default math mode, operands that TMA can map (16-byte base and
    row stride) or products of at least 2^24 multiply-adds (repacked first)
    take the tensor cores: 2-SM pairs from 256 units of work (256×256 tiles
    × 32-deep k-slices), except when at most 76 tiles of 128×128 and at
    most 32 k-slices (single blocks with split k); single blocks below;
  * otherwise the CUDA-core tile kernels: TMA-fed when both operands (as
    row-major copies for transposed ones) have 16-byte rows, or neither is
    transposed and the product has at least 2^32 multiply-adds (repacked
    first), and the stream-K iteration count fits 31 bits; else the
    any-layout kernel.
"""
import numpy as np
import pytest

import dense_fp32_matrix_gb300 as dfm


def tma_ok(addr, ld):
    return addr % 16 == 0 and (ld * 4) % 16 == 0 and ld * 4 < (1 << 40)


def model(op_a, op_b, M, N, K, lda, ldb, ldc, a, b, math):
    ta, tb = op_a == "T", op_b == "T"
    if M == 0 or N == 0 or K == 0:
        return "auto"
    if M == 1:
        return "gemv_col" if tb else "gemv_row"
    if N == 1:
        return "gemv_row" if (ta and ldc == 1 and (tb or ldb == 1)) \
            else "gemv_col"
    if M * N * K <= (1 << 23) and M <= 65535 * 32:
        return "small"
    aligned = tma_ok(a, lda) and tma_ok(b, ldb)
    if (aligned or M * N * K >= (1 << 24)) and math == "auto":
        work = -(-M // 256) * -(-N // 256) * -(-K // 32)
        tiles128 = -(-M // 128) * -(-N // 128)
        pair = work >= 256 and not (tiles128 <= 76 and -(-K // 32) <= 32)
        return "tf32x3_pair" if pair else "tf32x3"
    a_ok = K % 4 == 0 if ta else tma_ok(a, lda)
    b_ok = N % 4 == 0 if tb else tma_ok(b, ldb)
    repack = not ta and not tb and M * N * K >= (1 << 32)
    iters = -(-M // 256) * -(-N // 128) * -(-K // 32)
    return "tiled_tma" if (a_ok and b_ok or repack) and iters < (1 << 31) \
        else "tiled_ldg"


def _cases(n=600, seed=8080):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        M, N, K = (int(round(np.exp(rng.uniform(0.0, np.log(hi)))))
                   for hi in (20000, 20000, 20000))
        if rng.integers(8) == 0:
            M = 1
        if rng.integers(8) == 0:
            N = 1
        op_a, op_b = ("N", "T")[rng.integers(2)], ("N", "T")[rng.integers(2)]
        lda = (M if op_a == "T" else K) + int(rng.integers(0, 5))
        ldb = (K if op_b == "T" else N) + int(rng.integers(0, 5))
        ldc = N + int(rng.integers(0, 3)) if rng.integers(2) else max(N, 1)
        a = 0x7f0000000000 + 4 * int(rng.integers(0, 4))
        b = 0x7f4000000000 + 4 * int(rng.integers(0, 4))
        math = ("auto", "ffma")[rng.integers(2)]
        out.append((op_a, op_b, M, N, K, max(lda, 1), max(ldb, 1), ldc, a, b,
                    math))
    return out


@pytest.fixture(scope="module")
def lib():
    from dense_fp32_matrix_gb300 import build
    build.build()


def test_dispatch_matches_the_rules(lib):
    c_addr = 0x7f8000000000
    mismatches = []
    for case in _cases():
        op_a, op_b, M, N, K, lda, ldb, ldc, a, b, math = case
        prev = dfm.sgemm_set_math_mode(math)
        try:
            got = dfm.sgemm_plan_ex(op_a, op_b, M, N, K, lda, ldb, ldc, a, b,
                                    c_addr)
        finally:
            dfm.sgemm_set_math_mode(prev)
        want = model(*case)
        if got != want:
            mismatches.append((case, got, want))
    assert not mismatches, mismatches[:5]
