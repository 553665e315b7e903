"""Library calls captured into a CUDA graph replay to the same bits as the
direct calls (the per-device set-up and the stream's workspace are made by
a first call outside the capture, as the header asks)."""
import pytest

import matgen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_fp32_matrix_gb300 import build
    build.build()


def test_graph_replay_matches_direct_calls():
    import torch
    import dense_fp32_matrix_gb300 as dfm
    shapes = [(4096, 4096, 4096), (1024, 1024, 1024), (300, 260, 100),
              (1, 4096, 4096), (4095, 4097, 1023)]
    ops = []
    for i, (M, N, K) in enumerate(shapes):
        A = torch.from_numpy(matgen.uniform(30 + i, 0, M, K)).cuda()
        B = torch.from_numpy(matgen.uniform(30 + i, 1, K, N)).cuda()
        ops.append((M, N, K, A, B))
    s = torch.cuda.Stream()
    ref, out = [], []
    with torch.cuda.stream(s):
        for (M, N, K, A, B) in ops:            # direct calls (also warm-up)
            C = torch.empty(M, N, device="cuda")
            dfm.sgemm(M, N, K, A, K, B, N, C, N)
            ref.append(C)
        Ct = torch.empty(512, 512, device="cuda")
        Cb = torch.empty(3 * 256 * 256, device="cuda")
        Ab = torch.from_numpy(matgen.uniform(40, 0, 3 * 256, 128)).cuda()
        Bb = torch.from_numpy(matgen.uniform(40, 1, 3 * 128, 256)).cuda()
        At = torch.from_numpy(matgen.uniform(41, 0, 384, 512)).cuda()
        Bt = torch.from_numpy(matgen.uniform(41, 1, 512, 384)).cuda()
        Ct_ref = torch.empty(512, 512, device="cuda")
        Cb_ref = torch.empty_like(Cb)
        dfm.sgemm_ex("T", "T", 512, 512, 384, 1.5, At, 512, Bt, 384, 0.0,
                     Ct_ref, 512)
        dfm.sgemm_strided_batched("N", "N", 256, 256, 128, 1.0, Ab, 128,
                                  256 * 128, Bb, 256, 128 * 256, 0.0, Cb_ref,
                                  256, 256 * 256, 3)
        outs = [torch.full((M, N), float("nan"), device="cuda")
                for (M, N, K, A, B) in ops]
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for (M, N, K, A, B), C in zip(ops, outs):
            dfm.sgemm(M, N, K, A, K, B, N, C, N)
        dfm.sgemm_ex("T", "T", 512, 512, 384, 1.5, At, 512, Bt, 384, 0.0,
                     Ct, 512)
        dfm.sgemm_strided_batched("N", "N", 256, 256, 128, 1.0, Ab, 128,
                                  256 * 128, Bb, 256, 128 * 256, 0.0, Cb,
                                  256, 256 * 256, 3)
    for _ in range(3):
        for C in outs:
            C.fill_(float("nan"))
        Ct.fill_(float("nan"))
        Cb.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert dfm.sgemm_watchdog_status() == (0, 0)
        for C, R in zip(outs, ref):
            assert torch.equal(C, R)
        assert torch.equal(Ct, Ct_ref)
        assert torch.equal(Cb, Cb_ref)
