"""Seeded, counter-based synthetic matrices for the SGEMM path.

This module is the one piece shared by the CUDA path's tests/benchmark and the
CPU oracle: it produces input bits and nothing else. It holds none of the
matrix-product arithmetic.

The pages seed their inputs with a stateful generator (``torch.manual_seed(0)``
then ``torch.randn``, "GEMM from naive to tiled", section 11.2). A stateful
stream cannot be regenerated piecewise, so here every element is a pure
function of ``(seed, matrix_id, linear_index)``:

    key = seed * 2**40 + matrix_id * 2**36 + linear_index      (mod 2**64)
    h   = splitmix64(key)

``splitmix64`` is the published SplitMix64 step (Steele, Lea and Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014): add the
golden-ratio increment to the state, then apply the two xor-shift-multiply
rounds and a final xor-shift. ``linear_index = row * cols + col`` does not
depend on any leading dimension, so a padded copy holds the same values.

Distributions (all exactly representable in fp32):
  * ``uniform``:  ``(h >> 40) * 2**-23 - 1``, in [-1, 1), never 1.0;
  * ``integers``: ``((h >> 32) * 9) >> 32`` minus 4, in [-4, 4]
    (Lemire's multiply-shift range reduction);
  * ``normal``:   Box-Muller in fp64 from two hashes (index*2, index*2+1),
    rounded once to fp32.

matrix_id: A = 0, B = 1.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "splitmix64",
    "hash_keys",
    "uniform",
    "integers",
    "normal",
    "make",
    "KINDS",
    "MATRIX_A",
    "MATRIX_B",
]

MATRIX_A = 0
MATRIX_B = 1

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_MUL1 = np.uint64(0xBF58476D1CE4E5B9)
_MUL2 = np.uint64(0x94D049BB133111EB)


def splitmix64(state: np.ndarray) -> np.ndarray:
    """One SplitMix64 step applied elementwise to uint64 ``state``.

    Returns the output word for each state (the state advanced by the golden
    increment, then finalised). Wrapping uint64 arithmetic throughout.
    """
    z = np.asarray(state, dtype=np.uint64) + _GOLDEN
    z = (z ^ (z >> np.uint64(30))) * _MUL1
    z = (z ^ (z >> np.uint64(27))) * _MUL2
    return z ^ (z >> np.uint64(31))


def hash_keys(seed: int, matrix_id: int, idx: np.ndarray) -> np.ndarray:
    base = (int(seed) << 40) + (int(matrix_id) << 36)
    base &= (1 << 64) - 1
    with np.errstate(over="ignore"):
        return splitmix64(np.uint64(base) + np.asarray(idx, dtype=np.uint64))


def _linear(rows: int, cols: int) -> np.ndarray:
    return np.arange(rows * cols, dtype=np.uint64)


def uniform(seed: int, matrix_id: int, rows: int, cols: int) -> np.ndarray:
    """rows x cols fp32, i.i.d. uniform on [-1, 1) with 24-bit resolution."""
    h = hash_keys(seed, matrix_id, _linear(rows, cols))
    u = (h >> np.uint64(40)).astype(np.float64) * (2.0 ** -23) - 1.0
    return u.astype(np.float32).reshape(rows, cols)


def integers(seed: int, matrix_id: int, rows: int, cols: int) -> np.ndarray:
    """rows x cols fp32 holding integers uniform on [-4, 4]."""
    h = hash_keys(seed, matrix_id, _linear(rows, cols))
    hi = h >> np.uint64(32)
    with np.errstate(over="ignore"):
        v = (hi * np.uint64(9)) >> np.uint64(32)
    return (v.astype(np.int64) - 4).astype(np.float32).reshape(rows, cols)


def normal(seed: int, matrix_id: int, rows: int, cols: int) -> np.ndarray:
    """rows x cols fp32, i.i.d. standard normal by Box-Muller in fp64."""
    idx = _linear(rows, cols)
    with np.errstate(over="ignore"):
        h1 = hash_keys(seed, matrix_id, idx * np.uint64(2))
        h2 = hash_keys(seed, matrix_id, idx * np.uint64(2) + np.uint64(1))
    u1 = ((h1 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    u2 = (h2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)          # [0, 1)
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return z.astype(np.float32).reshape(rows, cols)


KINDS = {"uniform": uniform, "integers": integers, "normal": normal}


def make(kind: str, seed: int, matrix_id: int, rows: int, cols: int,
         ld: int | None = None, pad_value: float = np.nan) -> np.ndarray:
    """Generate a rows x cols matrix stored with leading dimension ``ld``.

    Returns an array of shape (rows, ld); columns ``cols..ld-1`` hold
    ``pad_value`` (NaN by default, so any read of the pitch padding by a
    kernel poisons its result). With ``ld`` None the array is dense.
    """
    m = KINDS[kind](seed, matrix_id, rows, cols)
    if ld is None or ld == cols:
        return m
    if ld < cols:
        raise ValueError("ld must be >= cols")
    out = np.full((rows, ld), pad_value, dtype=np.float32)
    out[:, :cols] = m
    return out
