"""Parity of sgemm_strided_batched with the CPU oracle, item by item.

Items are packed back to back without padding (stride = the item's size), so
a tile that read past an item's last row or k would pull in the next item's
numbers: every ragged tail is checked against the oracle of its own item."""
import numpy as np
import pytest

import matgen
import oracle
from gpu_util import compare

pytestmark = pytest.mark.gpu

OPS = [("N", "N"), ("N", "T"), ("T", "N"), ("T", "T")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_fp32_matrix_gb300 import build
    build.build()


def run_batch(ops, M, N, K, batch, alpha=1.0, beta=0.0, kind="uniform",
              seed=0, path="auto", shared_a=False, shared_b=False,
              side_by_side=False):
    import torch
    import dense_fp32_matrix_gb300 as dfm
    op_a, op_b = ops
    gen = matgen.KINDS[kind]
    na = 1 if shared_a else batch
    nb = 1 if shared_b else batch
    As = [gen(seed + 100 * b, 0, M, K) for b in range(na)]
    Bs = [gen(seed + 100 * b, 1, K, N) for b in range(nb)]
    A_st = [np.ascontiguousarray(a if op_a == "N" else a.T) for a in As]
    B_st = [np.ascontiguousarray(b if op_b == "N" else b.T) for b in Bs]
    lda, ldb = A_st[0].shape[1], B_st[0].shape[1]
    sa = 0 if shared_a else A_st[0].size
    sb = 0 if shared_b else B_st[0].size
    dA = torch.from_numpy(np.concatenate([a.ravel() for a in A_st])).cuda()
    dB = torch.from_numpy(np.concatenate([b.ravel() for b in B_st])).cuda()
    C0 = [gen(seed + 100 * b, 2, M, N) for b in range(batch)]
    if side_by_side:          # C as M x (batch * N): item b at column b * N
        ldc, sc = batch * N, N
        host = np.concatenate(C0, axis=1)
    else:
        ldc, sc = N, M * N
        host = np.concatenate([c.ravel() for c in C0])
    if beta == 0.0:
        host = np.full_like(host, np.nan)
    dC = torch.from_numpy(np.ascontiguousarray(host)).cuda()
    dfm.sgemm_strided_batched(op_a, op_b, M, N, K, alpha, dA, lda, sa, dB, ldb,
                              sb, beta, dC, ldc, sc, batch, path=path)
    torch.cuda.synchronize()
    assert dfm.sgemm_watchdog_status() == (0, 0)
    out = dC.cpu().numpy()
    for b in range(batch):
        if side_by_side:
            got = out.reshape(M, batch * N)[:, b * N:(b + 1) * N]
        else:
            got = out[b * M * N:(b + 1) * M * N].reshape(M, N)
        ref, S = oracle.gemm_ex(op_a, op_b, alpha, A_st[0 if shared_a else b],
                                B_st[0 if shared_b else b], beta,
                                None if beta == 0.0 else C0[b], M, N, K)
        compare(kind, got, ref, S, "batched item %d %s%s %s" % (
            b, op_a, op_b, path))


@pytest.mark.parametrize("path", ["auto", "tf32x3", "tf32x3_pair",
                                  "tiled_tma", "tiled_ldg"])
@pytest.mark.parametrize("ops", OPS, ids="".join)
def test_batched_packed_items(ops, path):
    run_batch(ops, 300, 260, 100, 3, kind="integers", seed=1, path=path)
    run_batch(ops, 300, 260, 100, 3, kind="uniform", seed=2, path=path)


@pytest.mark.parametrize("ops", OPS, ids="".join)
@pytest.mark.parametrize("shared", ["a", "b"])
@pytest.mark.parametrize("path", ["tf32x3_pair", "tiled_tma"])
def test_shared_operand(ops, shared, path):
    run_batch(ops, 264, 520, 132, 4, kind="integers", seed=3, path=path,
              shared_a=shared == "a", shared_b=shared == "b")


@pytest.mark.parametrize("ops", OPS, ids="".join)
def test_batched_scalars(ops):
    run_batch(ops, 200, 136, 72, 3, alpha=2.0, beta=-0.5, kind="integers",
              seed=4)
    run_batch(ops, 200, 136, 72, 3, alpha=-1.25, beta=0.75, kind="uniform",
              seed=5)
    run_batch(ops, 200, 136, 72, 3, alpha=0.0, beta=0.5, kind="integers",
              seed=6)


@pytest.mark.parametrize("ops", OPS, ids="".join)
def test_side_by_side_items(ops):
    run_batch(ops, 130, 64, 100, 4, kind="integers", seed=7,
              side_by_side=True)


def test_many_small_items_one_launch():
    run_batch(("N", "T"), 512, 512, 512, 16, kind="uniform", seed=8)
    run_batch(("N", "N"), 64, 64, 64, 40, kind="integers", seed=9)


def test_batch_of_one_matches_sgemm_ex_bitwise():
    import torch
    import dense_fp32_matrix_gb300 as dfm
    M, N, K = 1000, 1024, 600
    A = torch.from_numpy(matgen.uniform(10, 0, M, K)).cuda()
    B = torch.from_numpy(matgen.uniform(10, 1, K, N)).cuda()
    C1 = torch.empty(M, N, device="cuda")
    C2 = torch.empty(M, N, device="cuda")
    dfm.sgemm_ex("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C1, N)
    dfm.sgemm_strided_batched("N", "N", M, N, K, 1.0, A, K, 0, B, N, 0, 0.0,
                              C2, N, M * N, 1)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)


# A batch whose pair schedule has whole tiles and a stream-K tail (8 items
# of 4 x 4 tiles = 128 tiles on 76 clusters): the split tiles' pieces are
# summed under the whole tiles' MMAs and written straight to C, the whole
# tiles' accumulators are parked half in tensor memory; items of C stacked
# or side by side, with and without beta.
@pytest.mark.parametrize("side", [False, True])
@pytest.mark.parametrize("kind,alpha,beta", [("integers", 0.5, 2.0),
                                             ("uniform", 1.0, 0.0)])
def test_pair_batch_with_split_tail(side, kind, alpha, beta):
    run_batch(("N", "N"), 1024, 1024, 640, 8, alpha=alpha, beta=beta,
              kind=kind, seed=21, path="tf32x3_pair", side_by_side=side)


# Items side by side whose column offset (the item stride) is not a multiple
# of 4 floats while the row pitch is: item 1 starts 24 or 40 bytes into the
# row, so the kernels must fall back from 16-byte stores of C for every item.
@pytest.mark.parametrize("path", ["auto", "tf32x3", "tf32x3_pair"])
@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_side_by_side_item_stride_off_16_bytes(path, beta):
    run_batch(("N", "T"), 300, 6, 64, 2, beta=beta, kind="integers", seed=22,
              path=path, side_by_side=True)
    run_batch(("T", "T"), 132, 10, 36, 2, beta=beta, kind="uniform", seed=23,
              path=path, side_by_side=True)
