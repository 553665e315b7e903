"""Seeded random shapes through sgemm_ex on every 2-D path, each checked in
full against the CPU oracle (same bar as tests/test_ex_gpu.py: bit-exact on
integer data with power-of-two scalars, else |C - C_oracle| <= 1e-4 S +
1e-6). Sizes are log-uniform so that one-element edges, single tiles,
partial waves, stream-K tails (split tiles with whole tiles after them)
and ragged M, N, K all turn up; leading dimensions get random padding, so
misaligned rows (repacked for the tensor path) are covered too."""
import numpy as np
import pytest

from test_ex_gpu import run_ex

pytestmark = pytest.mark.gpu

PATHS = ["auto", "tf32x3_pair", "tf32x3", "tiled_tma", "tiled_ldg"]


def _cases(n=40, n_large=12, seed=20261202):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n + n_large:
        if len(out) < n:
            M, N, K = (int(round(np.exp(rng.uniform(0.0, np.log(hi)))))
                       for hi in (2600, 2900, 2100))
        else:  # several waves of 256 x 256 tiles: whole + split tiles
            M, N = (int(rng.integers(1500, 3100)) for _ in range(2))
            K = int(rng.integers(64, 1600))
        if M * N * K > 8e9:
            continue
        ops = ("N", "T")[rng.integers(2)], ("N", "T")[rng.integers(2)]
        kind = ("uniform", "integers")[rng.integers(2)]
        if kind == "integers":
            alpha, beta = [(1.0, 0.0), (0.5, 2.0), (-2.0, 1.0)][rng.integers(3)]
        else:
            alpha, beta = [(1.0, 0.0), (0.75, -1.5), (1.0, 1.0)][rng.integers(3)]
        path = PATHS[rng.integers(len(PATHS))]
        pad = int(rng.integers(0, 6))
        out.append((M, N, K, ops, kind, alpha, beta, path, pad,
                    int(rng.integers(1 << 20))))
    return out


CASES = _cases()


@pytest.mark.parametrize(
    "case", CASES,
    ids=["%dx%dx%d-%s%s-%s-%g-%g-%s-p%d" % (c[0], c[1], c[2], *c[3], c[4],
                                           c[5], c[6], c[7], c[8])
         for c in CASES])
def test_random_shapes(case):
    import dense_fp32_matrix_gb300 as dfm
    M, N, K, ops, kind, alpha, beta, path, pad, seed = case
    try:
        run_ex(*ops, M, N, K, alpha, beta, kind=kind, seed=seed, path=path,
               pad=pad)
    except dfm.SgemmError as e:
        # The TMA tile kernel needs 16-byte row strides for A and B (after
        # the row-major copy of a transposed operand); forcing it onto other
        # layouts is refused with SGEMM_ERR_PATH, never computed wrongly.
        if path == "tiled_tma" and e.status == dfm.STATUS["SGEMM_ERR_PATH"]:
            pytest.skip("tiled_tma refuses this layout")
        raise


def _batch_cases(n=20, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        M, N, K = (int(round(np.exp(rng.uniform(0.0, np.log(hi)))))
                   for hi in (700, 700, 600))
        batch = int(rng.integers(1, 6))
        if M * N * K * batch > 6e8:
            continue
        ops = ("N", "T")[rng.integers(2)], ("N", "T")[rng.integers(2)]
        kind = ("uniform", "integers")[rng.integers(2)]
        alpha, beta = [(1.0, 0.0), (0.5, 2.0)][rng.integers(2)]
        shared = int(rng.integers(3))  # 0 none, 1 A shared, 2 B shared
        side = bool(rng.integers(2))
        path = ("auto", "tf32x3_pair", "tiled_ldg")[rng.integers(3)]
        out.append((M, N, K, batch, ops, kind, alpha, beta, shared, side,
                    path, int(rng.integers(1 << 20))))
    return out


BATCH_CASES = _batch_cases()


@pytest.mark.parametrize(
    "case", BATCH_CASES,
    ids=["%dx%dx%dx%d-%s%s-%s-%g-%g-s%d-%s-%s" % (
        c[0], c[1], c[2], c[3], *c[4], c[5], c[6], c[7], c[8],
        "side" if c[9] else "stacked", c[10]) for c in BATCH_CASES])
def test_random_batches(case):
    from test_batched_gpu import run_batch
    M, N, K, batch, ops, kind, alpha, beta, shared, side, path, seed = case
    run_batch(ops, M, N, K, batch, alpha=alpha, beta=beta, kind=kind,
              seed=seed, path=path, shared_a=shared == 1,
              shared_b=shared == 2, side_by_side=side)


def _layout_cases(n=24, seed=4242):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        shape = rng.integers(4)
        M, N, K = (int(round(np.exp(rng.uniform(0.0, np.log(hi)))))
                   for hi in (3000, 3000, 3000))
        if shape == 0:
            M = 1
        elif shape == 1:
            N = 1
        if M * N * K > 3e9:
            continue
        pads = [int(rng.integers(0, 5)) for _ in range(3)]
        offs = tuple(int(rng.integers(0, 4)) for _ in range(3))
        out.append((M, N, K, pads, offs, ("uniform", "integers")[
            rng.integers(2)], int(rng.integers(1 << 20))))
    return out


LAYOUT_CASES = _layout_cases()


@pytest.mark.parametrize(
    "case", LAYOUT_CASES,
    ids=["%dx%dx%d-pad%s-off%s-%s" % (c[0], c[1], c[2], "".join(map(str, c[3])),
                                      "".join(map(str, c[4])), c[5])
         for c in LAYOUT_CASES])
def test_random_layouts(case):
    # sgemm (default dispatch) on pitched and misaligned operands: the
    # vector kernels, the repack before the tensor path, and the any-layout
    # tile kernel all get picked somewhere in here.
    from gpu_util import run_case
    M, N, K, pads, offs, kind, seed = case
    run_case(M, N, K, kind=kind, seed=seed, lda=max(K, 1) + pads[0],
             ldb=max(N, 1) + pads[1], ldc=max(N, 1) + pads[2], offsets=offs)


def _host_cases(n=12, seed=99):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        M, N, K = (int(round(np.exp(rng.uniform(0.0, np.log(hi)))))
                   for hi in (3000, 2500, 2000))
        if len(out) < 4:  # large enough for the row-block pipeline
            M, N, K = (int(rng.integers(512, 3000)),
                       int(rng.integers(600, 2500)),
                       int(rng.integers(1200, 2000)))
        if M * N * K > 8e9:
            continue
        pads = [int(rng.integers(0, 5)) for _ in range(3)]
        out.append((M, N, K, pads, ("uniform", "integers")[rng.integers(2)],
                    int(rng.integers(1 << 20))))
    return out


HOST_CASES = _host_cases()


@pytest.mark.parametrize(
    "case", HOST_CASES,
    ids=["%dx%dx%d-pad%s-%s" % (c[0], c[1], c[2], "".join(map(str, c[3])),
                                c[4]) for c in HOST_CASES])
def test_random_host_products(case):
    import torch
    import dense_fp32_matrix_gb300 as dfm
    import matgen
    import oracle
    from gpu_util import compare
    from test_host_pipeline_gpu import host_product
    M, N, K, pads, kind, seed = case
    A = matgen.KINDS[kind](seed, matgen.MATRIX_A, M, K)
    B = matgen.KINDS[kind](seed, matgen.MATRIX_B, K, N)
    hC, _ = host_product(A, B, M, N, K, *pads)
    torch.cuda.synchronize()
    assert dfm.sgemm_watchdog_status() == (0, 0)
    if pads[2]:
        assert torch.isnan(hC[:, N:]).all()      # pitch padding untouched
    ref, S = oracle.gemm(A, B)
    compare(kind, hC[:, :N].numpy(), ref, S, "sgemm_host %dx%dx%d" % (M, N, K))


def _noalloc_cases(n=12, seed=5150):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        M, N, K = (int(round(np.exp(rng.uniform(0.0, np.log(hi)))))
                   for hi in (3000, 3000, 2500))
        if M * N * K > 6e9:
            continue
        out.append((M, N, K, ("auto", "ffma")[rng.integers(2)],
                    ("uniform", "integers")[rng.integers(2)],
                    int(rng.integers(1 << 20))))
    return out


NOALLOC_CASES = _noalloc_cases()


@pytest.mark.parametrize(
    "case", NOALLOC_CASES,
    ids=["%dx%dx%d-%s-%s" % c[:5] for c in NOALLOC_CASES])
def test_random_noalloc(case):
    # the fixed-scratch entry point, in both math modes, against the oracle
    import torch
    import dense_fp32_matrix_gb300 as dfm
    import matgen
    import oracle
    from gpu_util import compare
    M, N, K, mode, kind, seed = case
    A_h = matgen.KINDS[kind](seed, matgen.MATRIX_A, M, K)
    B_h = matgen.KINDS[kind](seed, matgen.MATRIX_B, K, N)
    A = torch.from_numpy(A_h).cuda()
    B = torch.from_numpy(B_h).cuda()
    C = torch.full((M, N), float("nan"), device="cuda")
    prev = dfm.sgemm_set_math_mode(mode)
    try:
        dfm.sgemm_noalloc(M, N, K, A, max(K, 1), B, max(N, 1), C, max(N, 1))
        torch.cuda.synchronize()
    finally:
        dfm.sgemm_set_math_mode(prev)
    assert dfm.sgemm_watchdog_status() == (0, 0)
    ref, S = oracle.gemm(A_h, B_h)
    compare(kind, C.cpu().numpy(), ref, S, "sgemm_noalloc %dx%dx%d %s" % (
        M, N, K, mode))


def _mode_cases(n=16, seed=31337):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        if len(out) < 6:   # long k, few outputs: every tile split
            M, N = (int(round(np.exp(rng.uniform(0.0, np.log(700)))))
                    for _ in range(2))
            K = int(rng.integers(8000, 30000))
        else:
            M, N, K = (int(round(np.exp(rng.uniform(0.0, np.log(hi)))))
                       for hi in (2500, 2500, 2500))
        if M * N * K > 4e9:
            continue
        ops = ("N", "T")[rng.integers(2)], ("N", "T")[rng.integers(2)]
        kind = ("uniform", "integers")[rng.integers(2)]
        if kind == "integers":
            alpha, beta = [(1.0, 0.0), (0.5, 2.0)][rng.integers(2)]
        else:
            alpha, beta = [(1.0, 0.0), (0.75, -1.5)][rng.integers(2)]
        out.append((M, N, K, ops, kind, alpha, beta,
                    ("auto", "ffma")[rng.integers(2)],
                    int(rng.integers(0, 6)), int(rng.integers(1 << 20))))
    return out


MODE_CASES = _mode_cases()


@pytest.mark.parametrize(
    "case", MODE_CASES,
    ids=["%dx%dx%d-%s%s-%s-%g-%g-%s-p%d" % (c[0], c[1], c[2], *c[3], c[4],
                                           c[5], c[6], c[7], c[8])
         for c in MODE_CASES])
def test_random_math_modes(case):
    # default dispatch in both math modes (the CUDA-core kernels and the
    # vector kernels in "ffma"), including long-k products
    import dense_fp32_matrix_gb300 as dfm
    M, N, K, ops, kind, alpha, beta, mode, pad, seed = case
    prev = dfm.sgemm_set_math_mode(mode)
    try:
        run_ex(*ops, M, N, K, alpha, beta, kind=kind, seed=seed, pad=pad)
    finally:
        dfm.sgemm_set_math_mode(prev)
