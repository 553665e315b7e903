"""Synthetic workloads of the FP32 matrix-product path (shapes, value kinds,
seeds). Data only: no arithmetic of the product lives here.

Shapes follow the pages' problem size (M = N = K = 4096, "GEMM from naive to
tiled", section 二.1) widened to a square sweep, transformer-linear shapes,
and ragged / short-K / vector edge cases. Every float workload has an
integer-valued twin (entries uniform in [-4, 4]) whose product is exact in
fp32, for bit-exact comparison.
"""
from __future__ import annotations

FLOAT_WORKLOADS = (
    [dict(name="square_256", M=256, N=256, K=256, kind="uniform", seed=0),
     dict(name="square_4096", M=4096, N=4096, K=4096, kind="uniform", seed=1)]
    + [dict(name="square_%d" % s, M=s, N=s, K=s, kind="uniform", seed=s)
       for s in (512, 1024, 2048, 3072, 6144, 8192)]
    + [dict(name="linear_%dx%dx%d" % mnk, M=mnk[0], N=mnk[1], K=mnk[2],
            kind="normal", seed=2)
       for mnk in ((8192, 4096, 4096), (8192, 11008, 4096),
                   (8192, 4096, 11008))]
    + [dict(name="ragged_%dx%dx%d" % mnk, M=mnk[0], N=mnk[1], K=mnk[2],
            kind="uniform", seed=3)
       for mnk in ((4095, 4097, 1023), (4096, 4096, 64), (1, 4096, 4096),
                   (4096, 1, 4096), (127, 129, 33))]
)


def integer_twin(w: dict) -> dict:
    t = dict(w)
    t["name"] = w["name"] + "_int"
    t["kind"] = "integers"
    return t


WORKLOADS = FLOAT_WORKLOADS + [integer_twin(w) for w in FLOAT_WORKLOADS]

# The headline workload of the benchmark.
HEADLINE = FLOAT_WORKLOADS[1]


def by_name(name: str) -> dict:
    for w in WORKLOADS:
        if w["name"] == name:
            return dict(w)
    raise KeyError(name)
