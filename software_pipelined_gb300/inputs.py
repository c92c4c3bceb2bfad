"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no GEMM arithmetic: it only draws matrices.  It is the one
piece both the CUDA path's tests and the oracle's tests use, so it imports
neither of them.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; the 64-bit finaliser constants of Vigna's
public-domain splitmix64.c).  Output i (i = 0, 1, ...) of the stream seeded
with ``seed`` is mix(seed + (i+1)*0x9E3779B97F4A7C15) with
mix(z) = z3 ^ (z3 >> 31), z2 = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9,
z3 = (z2 ^ (z2 >> 27)) * 0x94D049BB133111EB, all mod 2^64.  Matrices are
filled in row-major order from one stream.

uniform[-1, 1):  u = (x >> 40) * 2^-23 - 1, i.e. 24 random bits; every value is
                 a multiple of 2^-23 and exactly representable in FP32.
normal N(0, 1):  Box-Muller in FP64 on consecutive output pairs (x0, x1):
                 u1 = ((x0 >> 11) + 1) * 2^-53 in (0, 1], u2 = (x1 >> 11) * 2^-53,
                 r = sqrt(-2 ln u1), values r*cos(2 pi u2), r*sin(2 pi u2),
                 then rounded to FP32.
"""
from __future__ import annotations

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

_CHUNK = 1 << 20


def _chunks(seed: int, n: int, start: int = 0):
    """Yield (offset, x) over outputs start .. start+n-1 of the stream, x a
    buffer of at most _CHUNK uint64 that is reused between chunks (every step
    in place, so long streams cost no allocation per chunk)."""
    s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    z = np.empty(min(n, _CHUNK), dtype=np.uint64)
    t = np.empty_like(z)
    with np.errstate(over="ignore"):
        for lo in range(0, n, _CHUNK):
            m = min(n, lo + _CHUNK) - lo
            x, y = z[:m], t[:m]
            x[:] = np.arange(start + lo + 1, start + lo + m + 1, dtype=np.uint64)
            np.multiply(x, GOLDEN_GAMMA, out=x)
            np.add(x, s, out=x)
            np.right_shift(x, np.uint64(30), out=y)
            np.bitwise_xor(x, y, out=x)
            np.multiply(x, _M1, out=x)
            np.right_shift(x, np.uint64(27), out=y)
            np.bitwise_xor(x, y, out=x)
            np.multiply(x, _M2, out=x)
            np.right_shift(x, np.uint64(31), out=y)
            np.bitwise_xor(x, y, out=x)
            yield lo, x


def splitmix64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs start .. start+n-1 of the SplitMix64 stream seeded with ``seed``."""
    out = np.empty(n, dtype=np.uint64)
    for lo, x in _chunks(seed, n, start):
        out[lo:lo + len(x)] = x
    return out


def uniform_pm1(seed: int, rows: int, cols: int, ld: int | None = None) -> np.ndarray:
    """rows x cols float32 matrix, i.i.d. uniform on [-1, 1) (24-bit grid).

    With ``ld`` > cols the result is a row-padded view of a rows x ld buffer
    whose padding holds NaN (so a reader that touches it is caught).
    """
    n = rows * cols
    v = np.empty(n, dtype=np.float32)
    f = np.empty(min(n, _CHUNK), dtype=np.float64)
    for lo, x in _chunks(seed, n):
        g = f[:len(x)]
        np.right_shift(x, np.uint64(40), out=x)
        g[:] = x
        np.multiply(g, 2.0 ** -23, out=g)
        np.subtract(g, 1.0, out=g)
        v[lo:lo + len(x)] = g
    return _place(v.reshape(rows, cols), ld)


def normal(seed: int, rows: int, cols: int, ld: int | None = None) -> np.ndarray:
    """rows x cols float32 matrix, i.i.d. N(0, 1) by FP64 Box-Muller."""
    n = rows * cols
    pairs = (n + 1) // 2
    z = np.empty(2 * pairs, dtype=np.float32)
    for lo, x in _chunks(seed, 2 * pairs):  # _CHUNK is even: chunks hold whole pairs
        u1 = ((x[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (x[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        r = np.sqrt(-2.0 * np.log(u1))
        t = 2.0 * np.pi * u2
        z[lo:lo + len(x):2] = r * np.cos(t)
        z[lo + 1:lo + len(x):2] = r * np.sin(t)
    return _place(z[:n].reshape(rows, cols), ld)


def small_int(seed: int, rows: int, cols: int, lo: int = -8, hi: int = 8,
              ld: int | None = None) -> np.ndarray:
    """Integers uniform on [lo, hi] stored as float32 (exact in TF32 and FP32)."""
    n = rows * cols
    span = np.uint64(hi - lo + 1)
    v = np.empty(n, dtype=np.float32)
    for c0, x in _chunks(seed, n):
        v[c0:c0 + len(x)] = ((x >> np.uint64(32)) % span).astype(np.int64) + lo
    return _place(v.reshape(rows, cols), ld)


def _bit_patterns(seed: int, rows: int, cols: int, lo: int, hi: int) -> np.ndarray:
    """float32 values whose magnitude bit pattern is uniform on [lo, hi)
    (integers), with a random sign (bit 0 of the same draw)."""
    n = rows * cols
    v = np.empty(n, dtype=np.uint32)
    span = np.uint64(hi - lo)
    for c0, x in _chunks(seed, n):
        mag = ((x >> np.uint64(32)) % span + np.uint64(lo)).astype(np.uint32)
        v[c0:c0 + len(x)] = mag | ((x & np.uint64(1)).astype(np.uint32) << np.uint32(31))
    return v.view(np.float32).reshape(rows, cols)


def top_of_range(seed: int, rows: int, cols: int) -> np.ndarray:
    """Finite values from the top 8192 FP32 magnitudes (bit patterns
    0x7F7FE000 .. 0x7F7FFFFF, about 3.4027e38 to FLT_MAX), random signs.  Half
    of them are at least 0x7F7FF000, where rounding to 10 mantissa bits
    would carry into the Inf exponent."""
    return _bit_patterns(seed, rows, cols, 0x7F7FE000, 0x7F800000)


def subnormal(seed: int, rows: int, cols: int) -> np.ndarray:
    """Nonzero FP32 subnormals (bit patterns 1 .. 0x7FFFFF: 2^-149 up to just
    below 2^-126), random signs."""
    return _bit_patterns(seed, rows, cols, 1, 0x00800000)


def scaled_exponents(seed: int, rows: int, cols: int, e_lo: int, e_hi: int) -> np.ndarray:
    """u * 2^e per element: u uniform on [-1, 1) (24-bit grid), e an integer
    uniform on [e_lo, e_hi] from the next draws of the same stream (so
    magnitudes span about 2^e_lo .. 2^e_hi).  Exact in FP32 as long as
    2^(e_lo - 23) is not below 2^-149."""
    u = uniform_pm1(seed, rows, cols).astype(np.float64)
    n = rows * cols
    span = np.uint64(e_hi - e_lo + 1)
    e = np.empty(n, dtype=np.float64)
    for c0, x in _chunks(seed, n, start=n):
        e[c0:c0 + len(x)] = ((x >> np.uint64(32)) % span).astype(np.int64) + e_lo
    return (u * np.exp2(e.reshape(rows, cols))).astype(np.float32)


def _place(M: np.ndarray, ld: int | None) -> np.ndarray:
    rows, cols = M.shape
    if ld is None or ld == cols:
        return M
    if ld < cols:
        raise ValueError("ld must be >= cols")
    buf = np.full((rows, ld), np.nan, dtype=np.float32)
    buf[:, :cols] = M
    return buf[:, :cols]


# Workloads of the pages' benchmark table and the large squares, with their
# seeds and distributions.  Each entry: (name, M, N, K, dist, seed_A, seed_B).
WORKLOADS = {
    "tiny_32": [("32x32x32", 32, 32, 32, "uniform", 1001, 1002)],
    "small_ragged": [
        ("128x128x128", 128, 128, 128, "uniform", 2001, 2002),
        ("512x512x512", 512, 512, 512, "uniform", 2003, 2004),
        ("127x193x61", 127, 193, 61, "uniform", 2005, 2006),
        ("513x257x129", 513, 257, 129, "uniform", 2007, 2008),
    ],
    "tall_skinny": [
        ("256x1024x128", 256, 1024, 128, "normal", 3001, 3002),
        ("1024x128x256", 1024, 128, 256, "normal", 3003, 3004),
    ],
    "square_1024": [("1024x1024x1024", 1024, 1024, 1024, "uniform", 4001, 4002)],
    "large_squares": [
        ("4096x4096x4096", 4096, 4096, 4096, "uniform", 5001, 5002),
        ("8192x8192x8192", 8192, 8192, 8192, "uniform", 5003, 5004),
    ],
}


def make_operands(M: int, N: int, K: int, dist: str, seed_a: int, seed_b: int,
                  lda: int | None = None, ldb: int | None = None):
    """A (M x K) and B (K x N) for one workload entry."""
    gen = {"uniform": uniform_pm1, "normal": normal, "int": small_int}[dist]
    return gen(seed_a, M, K, lda), gen(seed_b, K, N, ldb)
