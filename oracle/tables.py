"""Format constants of the oracle: TBQ sign vectors and Lloyd-Max centroid tables (16 levels
for TBQ4, 8 for turbo3).

KV cache math, "How a 4-bit cache gets away with it: rotate first": each 128-value block
is sign-flipped, Walsh-Hadamard transformed, sign-flipped again, and quantized with 16
Lloyd-Max centroids fitted to N(0, 1/sqrt(128)). The page fixes neither the sign seed nor
the table; the format fixes them here (sign words from splitmix64 at a stated seed; the
table by Lloyd iteration in fp64).
"""

import math
from functools import lru_cache

import numpy as np

MASK64 = (1 << 64) - 1
SIGN_SEED = 0x54425134
LLOYD_ITERS = 50_000


def splitmix64(state, n):
    """n outputs of splitmix64 (Steele, Lea & Flood 2014) from ``state``."""
    out = []
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        out.append(z ^ (z >> 31))
    return out


@lru_cache(maxsize=None)
def sign_words():
    return tuple(splitmix64(SIGN_SEED, 4))


@lru_cache(maxsize=None)
def tbq_signs():
    """(s1, s2) as float32 arrays of +-1, length 128: bit i of the words set -> -1."""
    w = sign_words()

    def expand(w0, w1):
        s = np.ones(128, dtype=np.float32)
        for i in range(128):
            word = w0 if i < 64 else w1
            if (word >> (i % 64)) & 1:
                s[i] = -1.0
        return s

    return expand(w[0], w[1]), expand(w[2], w[3])


def _phi(x):
    return math.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)


def _upper_tail(x):
    return 0.5 * math.erfc(x / math.sqrt(2.0))


def lloyd_max_gaussian(levels=16, iters=LLOYD_ITERS):
    """Ascending MSE-optimal levels for N(0,1), fp64, by Lloyd iteration.

    Symmetric: only the positive half is iterated. Cell k of the positive half is
    (b_k, b_{k+1}] with b_0 = 0, b_half = inf; its conditional mean is
    (phi(b_k) - phi(b_{k+1})) / (Q(b_k) - Q(b_{k+1})).
    """
    half = levels // 2
    c = [(k + 0.5) * 2.5 / half for k in range(half)]
    for _ in range(iters):
        b = [0.0] + [(c[k - 1] + c[k]) / 2.0 for k in range(1, half)] + [math.inf]
        new = []
        for k in range(half):
            lo, hi = b[k], b[k + 1]
            num = _phi(lo) - (0.0 if hi == math.inf else _phi(hi))
            den = _upper_tail(lo) - (0.0 if hi == math.inf else _upper_tail(hi))
            new.append(num / den)
        c = new
    return [-v for v in reversed(c)] + c


@lru_cache(maxsize=None)
def tbq4_tables():
    """(centroids[16], boundaries[15]) as float32 for N(0, sigma^2), sigma = 1/sqrt(128).

    boundaries[k-1] = beta_k = fp32(sigma * (C_{k-1} + C_k) / 2), k = 1..15.
    """
    sigma = 1.0 / math.sqrt(128.0)
    C = lloyd_max_gaussian(16)
    cent = np.array([sigma * v for v in C], dtype=np.float64).astype(np.float32)
    bnd = np.array([sigma * (C[k - 1] + C[k]) / 2.0 for k in range(1, 16)],
                   dtype=np.float64).astype(np.float32)
    return cent, bnd


@lru_cache(maxsize=None)
def tbq3_tables():
    """turbo3's (centroids[8], boundaries[7]) as float32, the same construction with 8 levels
    (the pages' turbo3 is the 3-bit relative of turbo4 = TBQ4: 50 B per 128 values)."""
    sigma = 1.0 / math.sqrt(128.0)
    C = lloyd_max_gaussian(8)
    cent = np.array([sigma * v for v in C], dtype=np.float64).astype(np.float32)
    bnd = np.array([sigma * (C[k - 1] + C[k]) / 2.0 for k in range(1, 8)], dtype=np.float64).astype(np.float32)
    return cent, bnd
