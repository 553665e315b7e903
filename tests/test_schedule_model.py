"""CPU model of the pair kernel's persistent schedule, checked for the
invariants the kernel relies on (no GPU).

The model restates, in Python, how the host plans a launch (whole tiles in
full waves, a stream-K tail split evenly over the clusters, every tile split
when tiles are fewer than clusters) and how each cluster walks its units
(its split share first, then its whole tiles). The invariants:

* every (tile, k-slice) is computed exactly once;
* a cluster's share holds at most two partial segments (the epilogue keeps
  room for two deferred fix-ups);
* a split tile's contributors are consecutive clusters in k order, so the
  pieces can be summed in cluster order;
* when a segment ends inside its tile and the cluster has whole tiles, the
  next unit is a whole tile (the fix-up summed early runs under its MMAs).

The GPU parity tests check the kernel itself on the same kinds of shapes.
"""
import pytest

TILE = 256        # pair tile, rows and columns
SLICE = 32        # k-slice depth
MIN_SK_SLICES = 8


def plan(M, N, K, clusters, batch=1):
    tiles = batch * (-(-M // TILE)) * (-(-N // TILE))
    T = -(-K // SLICE)
    G, dp, sk = min(tiles, clusters), tiles, 0
    rem = tiles % clusters
    if rem:
        if tiles < clusters:
            by_work = tiles * T // MIN_SK_SLICES if 4 * tiles <= 3 * clusters \
                else 0
            g = min(by_work, clusters)
            if g > tiles:
                G, sk, dp = g, tiles, 0
        else:
            s = rem
            if s * T // clusters < MIN_SK_SLICES:
                s += clusters
            if s * T // clusters >= MIN_SK_SLICES:
                G, sk, dp = clusters, s, tiles - s
    return dict(tiles=tiles, T=T, G=G, dp=dp, sk=sk, iters=sk * T)


def sk_begin(c, p):
    return c * p["iters"] // p["G"]


def units(c, p):
    """(tile, k_begin, k_end, split tile index or -1) in the cluster's order."""
    T, G = p["T"], p["G"]
    out = []
    if p["sk"]:
        b, e = sk_begin(c, p), sk_begin(c + 1, p)
        if b < e:
            for u in range((e - 1) // T - b // T + 1):
                x = b if u == 0 else (b // T + u) * T
                tau = x // T
                kb, ke = x - tau * T, min(e - tau * T, T)
                whole = kb == 0 and ke == T
                out.append((p["dp"] + tau, kb, ke, -1 if whole else tau))
    if c < p["dp"]:
        out += [(c + u * G, 0, T, -1) for u in range((p["dp"] - c + G - 1) // G)]
    return out


SHAPES = [(4096, 4096, 4096), (8192, 8192, 8192), (8192, 11008, 4096),
          (8192, 4096, 11008), (1792, 2816, 1024), (1000, 1000, 1000),
          (2048, 2048, 2048), (4096, 4096, 64), (2300, 2900, 1900),
          (20000, 260, 516), (1024, 1024, 4096), (4095, 4097, 1023),
          (256, 256, 32), (520, 780, 300), (6144, 6144, 6144)]


@pytest.mark.parametrize("clusters", [76, 64, 7, 1])
@pytest.mark.parametrize("shape", SHAPES, ids=str)
def test_schedule_invariants(shape, clusters):
    p = plan(*shape, clusters)
    T = p["T"]
    cover = {}
    contributors = {}
    for c in range(p["G"]):
        us = units(c, p)
        assert sum(1 for u in us if u[3] >= 0) <= 2
        for i, (tile, kb, ke, sk) in enumerate(us):
            assert 0 <= kb < ke <= T
            for k in range(kb, ke):
                cover[(tile, k)] = cover.get((tile, k), 0) + 1
            if sk >= 0:
                contributors.setdefault(tile, []).append((kb, c))
                if ke < T and c < p["dp"]:
                    assert i + 1 < len(us) and us[i + 1][3] < 0
    assert len(cover) == p["tiles"] * T
    assert all(v == 1 for v in cover.values())
    for tile, parts in contributors.items():
        parts.sort()
        clusters_in_k_order = [c for _, c in parts]
        assert clusters_in_k_order == list(range(clusters_in_k_order[0],
                                                 clusters_in_k_order[0] +
                                                 len(parts)))


def test_the_headline_schedule():
    # 4096^3 on 76 clusters: 228 whole tiles in three waves, the k-slices of
    # the last 28 tiles split 47.2 per cluster
    p = plan(4096, 4096, 4096, 76)
    assert (p["tiles"], p["T"], p["G"], p["dp"], p["sk"]) == (256, 128, 76,
                                                              228, 28)
    assert sum(len(units(c, p)) for c in range(76)) >= 228 + 28
