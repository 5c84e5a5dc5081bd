"""Floating-point helpers of the oracle (test infrastructure).

The codec arithmetic is fp32 with one IEEE rounding per operation; numpy's float32
ufuncs give exactly that. These helpers add the few conversions numpy lacks.
"""

import numpy as np

F32 = np.float32


def f32(x):
    return np.asarray(x, dtype=np.float32)


def to_f16(x):
    """fp32 -> fp16, round to nearest-even (numpy's cast), returned as float16."""
    return np.asarray(x, dtype=np.float32).astype(np.float16)


def f16_bits(h):
    return np.asarray(h, dtype=np.float16).view(np.uint16)


def bf16_bits_from_f32(x):
    """fp32 -> bf16 bit pattern, round to nearest-even, NaN kept quiet.

    A bf16 is the top 16 bits of an fp32. Rounding to nearest-even adds 0x7FFF plus the
    lowest kept bit before truncation.
    """
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) & np.uint64(0xFFFF)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    r = np.where(nan, (u >> np.uint64(16)) | np.uint64(0x40), r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def tree_sum(a, axis=-1):
    """Halving-tree sum along ``axis`` (length a power of two), fp32 adds.

    Each level adds the upper half onto the lower half: a[i] <- a[i] + a[i + n/2].
    """
    a = np.moveaxis(np.asarray(a, dtype=np.float32), axis, -1)
    n = a.shape[-1]
    assert n & (n - 1) == 0, "tree_sum needs a power-of-two length"
    while n > 1:
        n //= 2
        a = a[..., :n] + a[..., n:]
    return a[..., 0]
