"""Rotations of the oracle (test infrastructure).

SJ-KVaRN §2.2: each 256-value head vector is multiplied by an orthonormal 256-point
Hadamard matrix; 512-wide heads rotate each half on its own; queries are rotated the same
way and the attention output is rotated back. KV cache math, "rotate first": TBQ4 blocks
of 128 values are sign-flipped, Walsh-Hadamard transformed and sign-flipped again.

``fwht`` is the unnormalised Sylvester-order fast transform with ascending strides; it
works in the dtype it is given (fp32 for the codec, fp64 for the attention oracle).
"""

import numpy as np

from .tables import tbq_signs

NONE, HAD256, TBQ128 = "none", "had256", "tbq128"
TBQ_SCALE = np.float32(1.0 / np.sqrt(128.0))  # fp32(1/sqrt(128)) = 0x3DB504F3


def fwht(x):
    """Butterflies (a, b) -> (a + b, a - b) over pairs (i, i+s), s = 1, 2, 4, ..."""
    y = np.array(x, copy=True)
    n = y.shape[-1]
    s = 1
    while s < n:
        y = y.reshape(y.shape[:-1] + (n // (2 * s), 2, s))
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        y = y.reshape(y.shape[:-3] + (n,))
        s *= 2
    return y


def _blocks(x, n):
    x = np.asarray(x)
    assert x.shape[-1] % n == 0
    return x.reshape(x.shape[:-1] + (x.shape[-1] // n, n))


def rotate(x, kind):
    """fp32 forward rotation along the last axis (the codec-side rotation)."""
    x = np.asarray(x, dtype=np.float32)
    if kind == NONE:
        return x.copy()
    if kind == HAD256:
        y = fwht(_blocks(x, 256)) * np.float32(0.0625)
        return y.reshape(x.shape)
    if kind == TBQ128:
        s1, s2 = tbq_signs()
        y = fwht(_blocks(x, 128) * s1) * s2 * TBQ_SCALE
        return y.reshape(x.shape)
    raise ValueError(kind)


def rotate_f64(x, kind, inverse=False):
    """Exact orthonormal rotation in fp64 (attention oracle), forward or inverse."""
    x = np.asarray(x, dtype=np.float64)
    if kind == NONE:
        return x.copy()
    if kind == HAD256:
        return (fwht(_blocks(x, 256)) / 16.0).reshape(x.shape)
    if kind == TBQ128:
        s1, s2 = (a.astype(np.float64) for a in tbq_signs())
        if inverse:
            s1, s2 = s2, s1
        y = fwht(_blocks(x, 128) * s1) * s2 / np.sqrt(128.0)
        return y.reshape(x.shape)
    raise ValueError(kind)
