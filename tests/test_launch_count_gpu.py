"""The library counts the kernels it launches (sgemm_launch_count), and
bench.py reports that count as its gpu_launches claim. These tests pin the
count per call for each path: a path that quietly launched nothing, or more
kernels than it should, shows up here."""
import pytest

import matgen
import oracle
from gpu_util import compare, sample_indices

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_fp32_matrix_gb300 import build
    build.build()


# (M, N, K, math mode, expected plan, kernels per call)
CASES = [
    (1024, 1024, 1024, "ffma", "tiled_tma", 1),     # counters: a memset
    (1024, 1024, 1024, "auto", "tf32x3", 2),       # split k + reduce
    (2048, 2048, 2048, "auto", "tf32x3_pair", 1),
    (4095, 4097, 1023, "auto", "tf32x3_pair", 3),  # two repacks + pair
    (1, 4096, 1024, "auto", "gemv_row", 1),
    (1024, 1, 4096, "auto", "gemv_col", 1),
    (127, 129, 33, "auto", "small", 1),
    (2055, 2057, 1023, "ffma", "tiled_tma", 3),    # two repacks + tiles
]


@pytest.mark.parametrize("M,N,K,mode,plan,per_call", CASES)
def test_launches_per_call(M, N, K, mode, plan, per_call):
    import torch
    import dense_fp32_matrix_gb300 as dfm
    prev = dfm.sgemm_set_math_mode(mode)
    try:
        A_h = matgen.integers(71, matgen.MATRIX_A, M, K)
        B_h = matgen.integers(71, matgen.MATRIX_B, K, N)
        A, B = torch.from_numpy(A_h).cuda(), torch.from_numpy(B_h).cuda()
        C = torch.empty((M, N), device="cuda")
        got = dfm.sgemm_plan(M, N, K, K, N, N, A.data_ptr(), B.data_ptr(),
                             C.data_ptr())
        assert got == plan
        dfm.matmul(A, B, out=C)  # first call may allocate a workspace
        torch.cuda.synchronize()
        c0 = dfm.sgemm_launch_count()
        for _ in range(3):
            dfm.matmul(A, B, out=C)
        c1 = dfm.sgemm_launch_count()
        torch.cuda.synchronize()
        assert c1 - c0 == 3 * per_call
        assert dfm.sgemm_watchdog_status() == (0, 0)
        got_c = C.cpu().numpy()
        what = "%s %dx%dx%d" % (plan, M, N, K)
        if M * N * K <= 1 << 31:
            ref, S = oracle.gemm(A_h, B_h)
            compare("integers", got_c, ref, S, what)
        else:  # sampled rows of the oracle for the larger products
            rows, _, _ = sample_indices(M, N, rows=16)
            ref, S = oracle.gemm_rows(A_h, B_h, rows)
            compare("integers", got_c[rows], ref, S, what)
    finally:
        dfm.sgemm_set_math_mode(prev)


def test_rejected_call_launches_nothing():
    import torch
    import dense_fp32_matrix_gb300 as dfm
    A = torch.zeros((64, 64), device="cuda")
    c0 = dfm.sgemm_launch_count()
    with pytest.raises(dfm.SgemmError):
        # C overlaps A: refused on the host before anything is enqueued
        dfm.sgemm(64, 64, 64, A, 64, A, 64, A, 64)
    assert dfm.sgemm_launch_count() == c0
