"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle runs.

This module holds no step of the KV-cache method: it only draws the fp16 K/V/q values
that both the CUDA path and the CPU oracle consume, so that both see identical bytes.

Generator (counter-based, integer-only, so a CUDA kernel reproduces it bit for bit):

- ``mix64`` is the splitmix64 output function (Steele, Lea & Flood 2014).
- A stream is keyed by (seed, tensor, layer, seq, head) packed into 64 bits
  ``seed:8 | tensor:8 | layer:16 | seq:16 | head:16``; ``key = mix64(packed + GAMMA)``.
- Element ``i`` of a stream (``i = position * D + channel``) hashes to
  ``h = mix64(key + (i + 1) * GAMMA)``, i.e. the i-th splitmix64 output of that stream.
- The value is ``NORMAL_TABLE[h >> 48]``: a 65,536-entry table of fp16 standard-normal
  quantiles ``Phi^-1((j + 0.5) / 65536)``, so values are N(0,1) discretised at 2^-16
  probability steps, then rounded to fp16.
- Outlier channels (K only): ``n_out`` distinct channels per (layer, KV head), drawn from
  stream ``tensor = OUTLIER``; the K value there is ``fp16(fp32(x) * fp32(factor))``.
- Queries: ``fp16(fp32(x) * fp32(q_scale))`` with q_scale = 1/sqrt(head_dim) by default.

Tensor ids: K = 0, V = 1, Q = 2, OUTLIER = 3, CONTEXT = 4.
"""

from functools import lru_cache
from statistics import NormalDist

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB
MASK = (1 << 64) - 1
T_K, T_V, T_Q, T_OUTLIER, T_CONTEXT = 0, 1, 2, 3, 4


def mix64_int(z):
    z &= MASK
    z = ((z ^ (z >> 30)) * M1) & MASK
    z = ((z ^ (z >> 27)) * M2) & MASK
    return z ^ (z >> 31)


def mix64(z):
    """Vectorised mix64 over a uint64 numpy array (multiplication wraps mod 2^64)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(M2)
    return z ^ (z >> np.uint64(31))


def stream_key(seed, tensor, layer=0, seq=0, head=0):
    packed = ((seed & 0xFF) << 56) | ((tensor & 0xFF) << 48) | ((layer & 0xFFFF) << 32) \
        | ((seq & 0xFFFF) << 16) | (head & 0xFFFF)
    return mix64_int(packed + GAMMA)


@lru_cache(maxsize=None)
def normal_table():
    """65,536 fp16 quantiles of N(0,1) at probabilities (j + 0.5) / 65536."""
    nd = NormalDist()
    q = np.array([nd.inv_cdf((j + 0.5) / 65536.0) for j in range(65536)], dtype=np.float64)
    return q.astype(np.float16)


def stream_values(key, i0, n):
    """fp16 values of elements i0 .. i0+n-1 of the stream with key ``key``."""
    idx = np.arange(i0, i0 + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + (idx + np.uint64(1)) * np.uint64(GAMMA)
    h = mix64(z)
    return normal_table()[(h >> np.uint64(48)).astype(np.intp)]


def outlier_channels(seed, layer, head, head_dim, n_out):
    """n_out distinct channels in draw order from the OUTLIER stream of (layer, head)."""
    key = stream_key(seed, T_OUTLIER, layer, 0, head)
    out, j = [], 0
    while len(out) < n_out:
        c = mix64_int(key + (j + 1) * GAMMA) % head_dim
        if c not in out:
            out.append(c)
        j += 1
    return sorted(out)


def kv_values(seed, tensor, layer, seq, head, pos0, n_pos, head_dim, n_out=0, factor=1.0):
    """fp16 [n_pos, head_dim] for positions pos0.. of one (layer, seq, KV head)."""
    key = stream_key(seed, tensor, layer, seq, head)
    x = stream_values(key, pos0 * head_dim, n_pos * head_dim).reshape(n_pos, head_dim)
    if tensor == T_K and n_out > 0:
        ch = outlier_channels(seed, layer, head, head_dim, n_out)
        x = x.copy()
        x[:, ch] = (x[:, ch].astype(np.float32) * np.float32(factor)).astype(np.float16)
    return x


def kv_block(seed, tensor, layer, seq, pos0, n_pos, n_heads, head_dim, n_out=0, factor=1.0):
    """fp16 [n_pos, n_heads, head_dim] (the kv_append input layout)."""
    return np.stack([kv_values(seed, tensor, layer, seq, h, pos0, n_pos, head_dim, n_out, factor)
                     for h in range(n_heads)], axis=1)


def q_values(seed, layer, seq, step, n_q_heads, head_dim, q_scale=None):
    """fp16 [n_q_heads, head_dim] query of decode step ``step`` (stream position = step)."""
    s = np.float32(1.0 / np.sqrt(head_dim)) if q_scale is None else np.float32(q_scale)
    rows = []
    for h in range(n_q_heads):
        key = stream_key(seed, T_Q, layer, seq, h)
        x = stream_values(key, step * head_dim, head_dim)
        rows.append((x.astype(np.float32) * s).astype(np.float16))
    return np.stack(rows)


def context_lengths(seed, n, lo, hi):
    """n seeded lengths uniform in [lo, hi] (inclusive) from the CONTEXT stream."""
    key = stream_key(seed, T_CONTEXT)
    return [lo + mix64_int(key + (b + 1) * GAMMA) % (hi - lo + 1) for b in range(n)]
