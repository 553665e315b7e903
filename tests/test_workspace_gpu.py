"""Workspaces stay bounded when many short-lived streams call the library.

The stream-K and split-k paths keep their partial tiles in per-device
workspaces, one stream at a time, at most 8 of them. A stream that has none
while 8 exist takes the least recently used one after an event wait on the
device, so results stay those of the oracle even when the previous user's
kernels are still running."""
import pytest

import matgen
import oracle
from gpu_util import compare

pytestmark = pytest.mark.gpu

MAX_WORKSPACES = 8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_fp32_matrix_gb300 import build
    build.build()


@pytest.fixture(params=["auto", "ffma"])
def math_mode(request):
    # auto: 1024^3 takes single tensor blocks with split k (pieces in the
    # workspace); ffma: the stream-K tile kernel (partial tiles in it)
    import dense_fp32_matrix_gb300 as dfm
    previous = dfm.sgemm_set_math_mode(request.param)
    yield request.param
    dfm.sgemm_set_math_mode(previous)


def _operands(seed, M, N, K):
    import torch
    A_h = matgen.integers(seed, matgen.MATRIX_A, M, K)
    B_h = matgen.integers(seed, matgen.MATRIX_B, K, N)
    ref, S = oracle.gemm(A_h, B_h)
    return torch.from_numpy(A_h).cuda(), torch.from_numpy(B_h).cuda(), ref, S


def test_short_lived_streams_reuse_a_bounded_pool(math_mode):
    import torch
    import dense_fp32_matrix_gb300 as dfm
    M = N = K = 1024
    A, B, ref, S = _operands(61, M, N, K)
    sizes = []
    for i in range(3 * MAX_WORKSPACES):
        s = torch.cuda.Stream()
        C = torch.full((M, N), float("nan"), device="cuda")
        s.wait_stream(torch.cuda.current_stream())  # C filled, A, B copied
        dfm.matmul(A, B, out=C, stream=s)
        s.synchronize()
        compare("integers", C.cpu().numpy(), ref, S,
                "stream %d (%s)" % (i, math_mode))
        count, nbytes = dfm.sgemm_workspace_info()
        assert 1 <= count <= MAX_WORKSPACES
        sizes.append(nbytes)
        del s
    # once every workspace of the full pool has been handed over (and grown
    # to this size if an earlier caller left it smaller) it stops growing
    assert sizes[-1] == sizes[2 * MAX_WORKSPACES]
    assert dfm.sgemm_watchdog_status() == (0, 0)


def test_streams_in_flight_hand_over_workspaces(math_mode):
    # More streams than workspaces, all enqueued before any finishes: a
    # stream that takes another one's workspace must wait for that stream's
    # kernels on the device, or the partial tiles would mix.
    import torch
    import dense_fp32_matrix_gb300 as dfm
    M, N, K = 1024, 1024, 2048
    A, B, ref, S = _operands(62, M, N, K)
    streams = [torch.cuda.Stream() for _ in range(MAX_WORKSPACES + 5)]
    outs = [torch.full((M, N), float("nan"), device="cuda") for _ in streams]
    for s, C in zip(streams, outs):
        s.wait_stream(torch.cuda.current_stream())  # C filled, A, B copied
        dfm.matmul(A, B, out=C, stream=s)
    torch.cuda.synchronize()
    assert dfm.sgemm_watchdog_status() == (0, 0)
    for i, C in enumerate(outs):
        compare("integers", C.cpu().numpy(), ref, S,
                "in-flight stream %d (%s)" % (i, math_mode))
    count, _ = dfm.sgemm_workspace_info()
    assert count <= MAX_WORKSPACES
