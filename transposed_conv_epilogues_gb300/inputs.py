"""Seeded synthetic input generators shared by the tests, the bench and the oracle.

This module holds none of the method's arithmetic: it only turns a seed and an
element counter into fp32 numbers.  The generator is counter-based so that
any element can be regenerated independently:

* ``splitmix64`` (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): state_i = seed + (i + 1) * 0x9E3779B97F4A7C15,
  then the three xor-shift/multiply finalisation rounds.
* uniform in [0, 1): the top 53 bits of the splitmix64 output times 2^-53.
* standard normal: Box-Muller on the uniform pair drawn at counters 2i, 2i+1,
  r = sqrt(-2 ln(1 - u1)), z = r cos(2 pi u2).

The values are drawn in float64 and rounded once to float32; both the CUDA
path and the oracle consume the same float32 arrays.
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, counters: np.ndarray) -> np.ndarray:
    """splitmix64 output for each counter (uint64 array, wrap-around arithmetic)."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (counters.astype(np.uint64) + np.uint64(1)) * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """n float64 values in [0, 1) from counters offset .. offset+n-1."""
    c = np.arange(offset, offset + n, dtype=np.uint64)
    return (splitmix64(seed, c) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal(seed: int, shape, chunk: int = 1 << 24) -> np.ndarray:
    """Standard-normal float32 array of ``shape`` (Box-Muller, counters 2i, 2i+1)."""
    n = int(np.prod(shape))
    out = np.empty(n, np.float32)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        u = uniform01(seed, 2 * (e - s), 2 * s)
        r = np.sqrt(-2.0 * np.log1p(-u[0::2]))
        out[s:e] = (r * np.cos(2.0 * np.pi * u[1::2])).astype(np.float32)
    return out.reshape(shape)


def uniform(seed: int, shape, lo: float, hi: float, chunk: int = 1 << 24) -> np.ndarray:
    """float32 array of ``shape`` uniform in [lo, hi)."""
    n = int(np.prod(shape))
    out = np.empty(n, np.float32)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = (lo + (hi - lo) * uniform01(seed, e - s, s)).astype(np.float32)
    return out.reshape(shape)


def sample_indices(seed: int, total: int, count: int) -> np.ndarray:
    """``count`` distinct-ish flat indices in [0, total), sorted (for sampled parity checks)."""
    count = min(count, total)
    c = np.arange(count, dtype=np.uint64)
    v = splitmix64(seed, c) % np.uint64(total)
    return np.unique(v.astype(np.int64))
