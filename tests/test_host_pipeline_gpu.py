"""sgemm_host on products large enough to be pipelined: B, then row blocks
of A over the host link, each block of C computed as its rows land and
copied back while the next one computes. Parity with the CPU oracle, the
pitch padding of the host C left untouched, each row block equal to sgemm
of that block, and staging buffers reused by back-to-back calls."""
import numpy as np
import pytest

import matgen
import oracle
from gpu_util import compare, REL, ABS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_fp32_matrix_gb300 import build
    build.build()


@pytest.fixture(params=["auto", "ffma"])
def math_mode(request):
    import dense_fp32_matrix_gb300 as dfm
    prev = dfm.sgemm_set_math_mode(request.param)
    yield request.param
    dfm.sgemm_set_math_mode(prev)


def host_product(A, B, M, N, K, lda_pad=5, ldb_pad=3, ldc_pad=2, stream=None):
    """sgemm_host with pitched pinned host arrays; returns (hC view, hC)."""
    import torch
    import dense_fp32_matrix_gb300 as dfm
    hA = torch.full((M, K + lda_pad), float("nan")).pin_memory()
    hB = torch.full((K, N + ldb_pad), float("nan")).pin_memory()
    hA[:, :K] = torch.from_numpy(A)
    hB[:, :N] = torch.from_numpy(B)
    hC = torch.full((M, N + ldc_pad), float("nan")).pin_memory()
    dA = torch.empty(M * K, device="cuda")
    dB = torch.empty(K * N, device="cuda")
    dC = torch.empty(M * N, device="cuda")
    dfm.sgemm_host(M, N, K, hA, K + lda_pad, hB, N + ldb_pad, hC, N + ldc_pad,
                   dA, dB, dC, stream)
    return hC, (dA, dB, dC)


@pytest.mark.parametrize("mnk", [(2048, 1024, 1024), (1000, 2300, 1100),
                                 (1536, 1100, 1300)], ids=str)
@pytest.mark.parametrize("kind", ["uniform", "integers"])
def test_pipelined_host_product(mnk, kind, math_mode):
    import torch
    import dense_fp32_matrix_gb300 as dfm
    M, N, K = mnk
    A = matgen.KINDS[kind](21, matgen.MATRIX_A, M, K)
    B = matgen.KINDS[kind](21, matgen.MATRIX_B, K, N)
    hC, _ = host_product(A, B, M, N, K)
    torch.cuda.synchronize()
    assert dfm.sgemm_watchdog_status() == (0, 0)
    assert torch.isnan(hC[:, N:]).all()          # pitch padding untouched
    got = hC[:, :N].numpy()
    ref, S = oracle.gemm(A, B, M=M, N=N, K=K, lda=K, ldb=N)
    compare(kind, got, ref, S, "sgemm_host %dx%dx%d %s" % (M, N, K, kind))


def test_each_row_block_is_sgemm_of_that_block():
    # 4 blocks of 512 rows for M = 2048; each equals sgemm of its rows.
    import torch
    import dense_fp32_matrix_gb300 as dfm
    M, N, K = 2048, 1024, 1024
    A = matgen.normal(22, matgen.MATRIX_A, M, K)
    B = matgen.normal(22, matgen.MATRIX_B, K, N)
    hC, _ = host_product(A, B, M, N, K)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    blocks = [dfm.matmul(dA[r:r + 512], dB) for r in range(0, M, 512)]
    torch.cuda.synchronize()
    assert torch.equal(hC[:, :N], torch.cat(blocks).cpu())


def test_back_to_back_calls_reuse_staging_buffers():
    # The second call's copies must not overwrite the staging buffers before
    # the first call's products and copy-back are done.
    import torch
    import dense_fp32_matrix_gb300 as dfm
    M, N, K = 2048, 1024, 1024
    A1 = matgen.uniform(23, matgen.MATRIX_A, M, K)
    A2 = matgen.uniform(24, matgen.MATRIX_A, M, K)
    B = matgen.uniform(23, matgen.MATRIX_B, K, N)
    hB = torch.from_numpy(B).pin_memory()
    dA = torch.empty(M * K, device="cuda")
    dB = torch.empty(K * N, device="cuda")
    dC = torch.empty(M * N, device="cuda")
    outs = []
    for A in (A1, A2, A1):
        hA = torch.from_numpy(A).pin_memory()
        hC = torch.empty((M, N)).pin_memory()
        dfm.sgemm_host(M, N, K, hA, K, hB, N, hC, N, dA, dB, dC)
        outs.append((A, hC))
    torch.cuda.synchronize()
    for A, hC in outs:
        ref, S = oracle.gemm(A, B, M=M, N=N, K=K, lda=K, ldb=N)
        err = np.abs(hC.numpy().astype(np.float64) - ref)
        assert np.all(err <= REL * S + ABS)
    assert torch.equal(outs[0][1], outs[2][1])
