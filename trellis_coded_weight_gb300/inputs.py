"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module draws random numbers and rounds them to the storage types of the
inputs (bf16, fp16, uint32).  It holds none of the trellis method's arithmetic:
no window extraction, no 1MAD code, no scaling, no matvec.  Both the CUDA path
and the oracle receive the arrays it returns.

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014), one independent stream per tensor, keyed by a seed.
Uniform doubles take the top 53 bits; normals use the Box-Muller transform.

Input recipe (the workloads are the ~27B-class MLP projection shapes, hidden
5120 / intermediate 17408):
  * codes   uniform random 32-bit words (every bitstream is a valid tail-biting
            trellis path, so uniform words are valid codes)
  * scales  U[0.005, 0.02] drawn in double, rounded to fp16 (round-to-nearest-even)
  * x       N(0, sigma) drawn in double, rounded to fp32 then to bf16 (RNE)
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Default seeds, one stream per tensor role.
SEED_CODES = 1001
SEED_GATE = 1002
SEED_UP = 1003
SEED_SCALES = 2001
SEED_X = 3001


def splitmix64(seed: int, n: int) -> np.ndarray:
    """Return n consecutive SplitMix64 outputs of the stream keyed by ``seed``."""
    with np.errstate(over="ignore"):
        idx = np.arange(1, n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, n: int) -> np.ndarray:
    """n doubles uniform in [0, 1) from the top 53 bits of SplitMix64."""
    return (splitmix64(seed, n) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def random_words(seed: int, shape) -> np.ndarray:
    """Uniform random uint32 words (two per 64-bit draw), C-contiguous."""
    n = int(np.prod(shape))
    draws = splitmix64(seed, (n + 1) // 2)
    words = draws.view(np.uint32)[:n]
    return np.ascontiguousarray(words.reshape(shape))


def _f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 storage bits, nearest-even (inputs are finite)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep = u >> np.uint64(16)
    rest = u & np.uint64(0xFFFF)
    up = (rest > 0x8000) | ((rest == 0x8000) & ((keep & np.uint64(1)) == 1))
    return (keep + up.astype(np.uint64)).astype(np.uint16)


def normal_bf16(seed: int, shape, sigma: float = 1.0) -> np.ndarray:
    """bf16 storage bits (uint16) of N(0, sigma) draws (Box-Muller, double)."""
    n = int(np.prod(shape))
    m = (n + 1) // 2
    u = uniform01(seed, 2 * m)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log1p(-u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    z = (sigma * z[:n]).astype(np.float32)
    return _f32_to_bf16_bits(z).reshape(shape)


def uniform_f16(seed: int, shape, lo: float = 0.005, hi: float = 0.02) -> np.ndarray:
    """fp16 storage bits (uint16) of U[lo, hi] draws (double, then RNE to fp16)."""
    n = int(np.prod(shape))
    v = lo + (hi - lo) * uniform01(seed, n)
    return v.astype(np.float16).view(np.uint16).reshape(shape)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 storage bits to fp32 values (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen fp16 storage bits to fp32 values (exact)."""
    return np.asarray(b, dtype=np.uint16).view(np.float16).astype(np.float32)


def words_per_row(cols: int, k: int) -> int:
    return cols * k // 32


def make_linear(rows: int, cols: int, k: int, M: int, *, seed_codes: int = SEED_CODES,
                seed_scales: int = SEED_SCALES, seed_x: int = SEED_X, sigma: float = 1.0,
                x_len: int | None = None):
    """Codes [rows, cols*k/32] uint32, scales [rows] fp16 bits, x [M, x_len] bf16 bits.

    ``x_len`` defaults to ``cols`` (axis-1 layers); axis-0 layers pass ``rows``.
    """
    codes = random_words(seed_codes, (rows, words_per_row(cols, k)))
    scales = uniform_f16(seed_scales, (rows,))
    x = normal_bf16(seed_x, (M, cols if x_len is None else x_len), sigma)
    return codes, scales, x
