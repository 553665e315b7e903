"""The FFMA tile kernel's schedule, modelled on the CPU (no GPU).

The kernel deals whole 256 x 128 tiles in full waves (tile t to block
t mod G) and splits the k-slices of the remaining tiles evenly over all G
blocks (stream-K), one more wave being split when a share would be under 8
k-slices. Each block walks its split share first (a partial segment at
either end, whole tiles between), then its whole tiles. A partial segment
is a piece in the workspace slot 2b (the share's first segment) or 2b + 1
(its last); the last block to arrive on a split tile finds every piece
from the blocks that cover the tile. This model restates those rules and
checks, over seeded shapes and grid sizes, that every (tile, k-slice) is
computed exactly once, that each tile is written once (whole or from its
pieces), that the pieces found cover the tile's k-slices once in k order,
and that slots and counters stay inside their buffers."""
import numpy as np
import pytest

BM, BN, BK, WARPS, MIN_SHARE = 256, 128, 32, 8, 8


def plan(M, N, K, resident):
    tiles = -(-M // BM) * -(-N // BN)
    iters = -(-K // BK)
    total = tiles * iters
    grid = max(1, min(resident, total))
    waves = tiles // grid
    rest = tiles - waves * grid
    if waves > 0 and rest > 0 and rest * iters < MIN_SHARE * grid:
        waves -= 1
    dp = waves * grid
    return dict(tiles=tiles, I=iters, G=grid, dp=dp, sk=(tiles - dp) * iters,
                counters=(tiles - dp) * WARPS, ws_slots=2 * grid)


def segments(p, b):
    I, G, dp, sk = p["I"], p["G"], p["dp"], p["sk"]
    x, x_end = b * sk // G, (b + 1) * sk // G
    out = []
    while x < x_end:
        t = x // I
        end = min(x_end, (t + 1) * I)
        out.append((dp + t, x - t * I, end - x))
        x = end
    out += [(t, 0, I) for t in range(b, dp, G)]
    return out


def check(M, N, K, resident):
    p = plan(M, N, K, resident)
    I, G, dp, sk = p["I"], p["G"], p["dp"], p["sk"]
    begin = lambda c: c * sk // G
    owner = lambda x: ((x + 1) * G + sk - 1) // sk - 1
    done = np.zeros((p["tiles"], I), dtype=np.int64)
    written, pieces = {}, {}
    for b in range(G):
        for n, (tile, kt0, ln) in enumerate(segments(p, b)):
            done[tile, kt0:kt0 + ln] += 1
            if kt0 == 0 and ln == I:
                assert tile not in written
                written[tile] = "whole"
            else:
                assert tile >= dp
                slot = 2 * b + (0 if n == 0 else 1)
                assert slot < p["ws_slots"] and slot not in pieces
                assert (tile - dp + 1) * WARPS <= p["counters"]
                pieces[slot] = (tile, kt0, ln)
    assert (done == 1).all()
    for tile in range(dp, p["tiles"]):
        if tile in written:
            continue
        x0 = (tile - dp) * I
        ks = []
        for c in range(owner(x0), owner(x0 + I - 1) + 1):
            t, kt0, ln = pieces[2 * c + (0 if begin(c) >= x0 else 1)]
            assert t == tile
            ks += list(range(kt0, kt0 + ln))
        assert ks == list(range(I))
        written[tile] = "pieces"
    assert len(written) == p["tiles"]
    return p


@pytest.mark.parametrize("resident", [152, 160, 1, 7])
def test_schedule_random_shapes(resident):
    rng = np.random.default_rng(1000 + resident)
    for _ in range(150):
        M, N = (int(round(np.exp(rng.uniform(0, np.log(20000))))) for _ in "MN")
        K = int(round(np.exp(rng.uniform(0, np.log(9000)))))
        check(M, N, K, resident)


def test_schedule_of_the_workloads():
    # 4096^3: three whole waves (456 tiles), 56 tiles split over 152 blocks
    p = check(4096, 4096, 4096, 152)
    assert (p["dp"], p["sk"]) == (456, 56 * 128)
    # fewer tiles than blocks: every tile split
    p = check(2048, 2048, 2048, 152)
    assert (p["dp"], p["sk"]) == (0, 128 * 64)
    # a share under 8 k-slices takes one more wave
    p = check(8192, 11008, 4096, 152)
    assert p["sk"] // p["G"] >= MIN_SHARE
    for mnk in [(8192, 8192, 8192), (8192, 4096, 11008), (4096, 4096, 64),
                (4095, 4097, 1023), (256 * 153, 128, 4)]:
        check(*mnk, 152)
