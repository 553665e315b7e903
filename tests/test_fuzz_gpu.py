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
