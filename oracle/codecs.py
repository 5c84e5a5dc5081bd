"""Block codecs of the oracle (test infrastructure): tq6_0, TBQ4, Q8_0, Q4_0, Q5_0, Q6_0,
Q4_1, Q5_1.

All encoders take fp32 values whose last axis is a whole number of blocks and return
(scale fp16 array, code array of small integers); packers turn code arrays into the
stored bytes. Arithmetic: one IEEE fp32 rounding per operation, numpy's ``rint``
(half to even), fp16 by round-to-nearest-even.

Sources:
- tq6_0: SJ-KVaRN §2.1 item 2 ("rotated 6-bit format: 98 bytes per 128 values").
- TBQ4: KV cache math, "Worked example" (66 B = 2-byte scale + 64 B of 4-bit indices per
  128 values) and "rotate first" (16 Lloyd-Max centroids, one FP16 norm per block).
- Q8_0 (34 B / 32) and Q4_0 (18 B / 32): KV cache math, the format table; HAL #582 §1.
"""

import numpy as np

from .fp import f32, to_f16, tree_sum
from . import tables
from .tables import tbq4_tables


def _blocks(x, n):
    x = f32(x)
    assert x.shape[-1] % n == 0
    return x.reshape(x.shape[:-1] + (x.shape[-1] // n, n))


# ----------------------------------------------------------------------------- tq6_0
def tq6_encode(x):
    """x[..., 128k] -> (d fp16 [..., k], code uint8 [..., k, 128] in 1..63)."""
    xb = _blocks(x, 128)
    a = np.max(np.abs(xb), axis=-1)
    d = to_f16(a / np.float32(31.0))
    d32 = d.astype(np.float32)
    zero = d32 == 0
    with np.errstate(divide="ignore"):
        inv = np.where(zero, np.float32(0), np.float32(1.0) / np.where(zero, np.float32(1), d32))
    q = np.rint(xb * inv[..., None].astype(np.float32))
    q = np.clip(q, -31, 31)
    q = np.where(zero[..., None], 0, q)
    return d, (q + 32).astype(np.uint8)


def tq6_decode(d, code):
    return ((code.astype(np.float32) - np.float32(32)) * d.astype(np.float32)[..., None]).reshape(
        code.shape[:-2] + (code.shape[-2] * 128,))


def tq6_pack(code):
    """code [..., 128] (6-bit) -> (ql [..., 64], qh [..., 32]) uint8."""
    c = code.astype(np.uint8)
    lo = c & 0x0F
    hi = (c >> 4) & 0x03
    ql = (lo[..., 0::2] | (lo[..., 1::2] << 4)).astype(np.uint8)
    qh = (hi[..., 0::4] | (hi[..., 1::4] << 2) | (hi[..., 2::4] << 4) | (hi[..., 3::4] << 6)).astype(np.uint8)
    return ql, qh


def tq6_unpack(ql, qh):
    lo = np.empty(ql.shape[:-1] + (128,), dtype=np.uint8)
    lo[..., 0::2] = ql & 0x0F
    lo[..., 1::2] = ql >> 4
    hi = np.empty_like(lo)
    for m in range(4):
        hi[..., m::4] = (qh >> (2 * m)) & 0x03
    return (lo | (hi << 4)).astype(np.uint8)


# ----------------------------------------------------------------------------- TBQ4
def tbq4_encode(y):
    """y[..., 128k] (rotated) -> (n16 fp16 [..., k], idx uint8 [..., k, 128] in 0..15)."""
    cent, bnd = tbq4_tables()
    yb = _blocks(y, 128)
    ss = tree_sum(yb * yb, axis=-1)
    n16 = to_f16(np.sqrt(ss))
    n32 = n16.astype(np.float32)
    zero = n32 == 0
    inv = np.where(zero, np.float32(0), np.float32(1.0) / np.where(zero, np.float32(1), n32))
    u = yb * inv[..., None].astype(np.float32)
    idx = np.zeros(u.shape, dtype=np.uint8)
    for k in range(15):
        idx += (u > bnd[k]).astype(np.uint8)
    return n16, idx


def turbo3_encode(y):
    """The pages' turbo3 (SJ-KVaRN §2.1, §7.2: a rotated 3-bit format, 50 B per 128 values),
    read as TBQ4 with 8 levels: y[..., 128k] (rotated) -> (n16 fp16 [..., k], idx [..., k, 128]
    in 0..7), idx = #{k : u > beta_k} with u = y / fp32(n16)."""
    cent, bnd = tables.tbq3_tables()
    yb = _blocks(y, 128)
    ss = tree_sum(yb * yb, axis=-1)
    n16 = to_f16(np.sqrt(ss))
    n32 = n16.astype(np.float32)
    zero = n32 == 0
    inv = np.where(zero, np.float32(0), np.float32(1.0) / np.where(zero, np.float32(1), n32))
    u = yb * inv[..., None].astype(np.float32)
    idx = np.zeros(u.shape, dtype=np.uint8)
    for k in range(7):
        idx += (u > bnd[k]).astype(np.uint8)
    return n16, idx


def turbo3_decode(n16, idx):
    cent, _ = tables.tbq3_tables()
    v = cent[idx] * n16.astype(np.float32)[..., None]
    return v.reshape(idx.shape[:-2] + (idx.shape[-2] * 128,))


def tq5_encode(y):
    """The pages' tq5_0 (a rotated 5-bit format, 82 B per 128 values), read like tq6_0 with 15
    levels a side: y[..., 128k] -> (d fp16 [..., k], code [..., k, 128] in 1..31; 16 is zero)."""
    yb = _blocks(y, 128)
    d = to_f16(np.max(np.abs(yb), axis=-1) / np.float32(15.0))
    d32 = d.astype(np.float32)
    zero = d32 == 0
    inv = np.where(zero, np.float32(0), np.float32(1.0) / np.where(zero, np.float32(1), d32))
    q = np.clip(np.rint(yb * inv[..., None].astype(np.float32)), -15, 15)
    return d, (q + 16).astype(np.uint8)


def tq5_decode(d, code):
    v = (code.astype(np.float32) - np.float32(16)) * d.astype(np.float32)[..., None]
    return v.reshape(code.shape[:-2] + (code.shape[-2] * 128,))


def tbq4_decode(n16, idx):
    cent, _ = tbq4_tables()
    v = cent[idx.astype(np.intp)] * n16.astype(np.float32)[..., None]
    return v.reshape(idx.shape[:-2] + (idx.shape[-2] * 128,))


# ----------------------------------------------------------------------------- Q8_0 / Q4_0
def q8_encode(x):
    """x[..., 32k] -> (d fp16 [..., k], q int8 [..., k, 32])."""
    xb = _blocks(x, 32)
    d = to_f16(np.max(np.abs(xb), axis=-1) / np.float32(127.0))
    d32 = d.astype(np.float32)
    zero = d32 == 0
    inv = np.where(zero, np.float32(0), np.float32(1.0) / np.where(zero, np.float32(1), d32))
    q = np.clip(np.rint(xb * inv[..., None].astype(np.float32)), -127, 127)
    return d, q.astype(np.int8)


def q8_decode(d, q):
    v = q.astype(np.float32) * d.astype(np.float32)[..., None]
    return v.reshape(q.shape[:-2] + (q.shape[-2] * 32,))


def q4_encode(x):
    """x[..., 32k] -> (d fp16 [..., k], code uint8 [..., k, 32] in 1..15; 8 is zero)."""
    xb = _blocks(x, 32)
    d = to_f16(np.max(np.abs(xb), axis=-1) / np.float32(7.0))
    d32 = d.astype(np.float32)
    zero = d32 == 0
    inv = np.where(zero, np.float32(0), np.float32(1.0) / np.where(zero, np.float32(1), d32))
    q = np.clip(np.rint(xb * inv[..., None].astype(np.float32)), -7, 7)
    return d, (q + 8).astype(np.uint8)


def q4_decode(d, code):
    v = (code.astype(np.float32) - np.float32(8)) * d.astype(np.float32)[..., None]
    return v.reshape(code.shape[:-2] + (code.shape[-2] * 32,))


# ----------------------------------------------------------------------------- Q5_0 / Q6_0 / Q4_1 / Q5_1
# The other 32-value block formats the pages compare against (SJ-KVaRN §4.1, §6: q5_1 "a 5-bit
# block format with a scale and an offset", 24 B / 32; KV cache math and the Qwen page: q5_0
# 22 B, q6_0 26 B, q4_1 20 B per 32). Reading (the pages give only sizes and names): the _0
# formats are symmetric like Q4_0, d = fp16(max|x| / L), code = clamp(rint(x / d), -L, L) + L + 1
# (L = 15, 31); the _1 formats take the block's minimum as the offset, m = fp16(min x),
# d = fp16((max x - min x) / Q), code = clamp(rint((x - m) / d), 0, Q) (Q = 15, 31), d = 0 -> 0.
def qsym_encode(x, L):
    """x[..., 32k] -> (d fp16 [..., k], code uint8 [..., k, 32] in 1..2L+1; L+1 is zero)."""
    xb = _blocks(x, 32)
    d = to_f16(np.max(np.abs(xb), axis=-1) / np.float32(L))
    d32 = d.astype(np.float32)
    zero = d32 == 0
    inv = np.where(zero, np.float32(0), np.float32(1.0) / np.where(zero, np.float32(1), d32))
    q = np.clip(np.rint(xb * inv[..., None].astype(np.float32)), -L, L)
    return d, (q + (L + 1)).astype(np.uint8)


def qsym_decode(d, code, L):
    v = (code.astype(np.float32) - np.float32(L + 1)) * d.astype(np.float32)[..., None]
    return v.reshape(code.shape[:-2] + (code.shape[-2] * 32,))


def qmin_encode(x, Q):
    """x[..., 32k] -> (d fp16, m fp16 [..., k], code uint8 [..., k, 32] in 0..Q)."""
    xb = _blocks(x, 32)
    lo = np.min(xb, axis=-1)
    hi = np.max(xb, axis=-1)
    m = to_f16(lo)
    d = to_f16((hi - lo) / np.float32(Q))
    d32, m32 = d.astype(np.float32), m.astype(np.float32)
    zero = d32 == 0
    inv = np.where(zero, np.float32(0), np.float32(1.0) / np.where(zero, np.float32(1), d32))
    with np.errstate(invalid="ignore"):
        q = np.clip(np.rint((xb - m32[..., None]) * inv[..., None].astype(np.float32)), 0, Q)
    q = np.where(zero[..., None], 0, q)
    return d, m, q.astype(np.uint8)


def qmin_decode(d, m, code):
    v = code.astype(np.float32) * d.astype(np.float32)[..., None] + m.astype(np.float32)[..., None]
    return v.reshape(code.shape[:-2] + (code.shape[-2] * 32,))


# ----------------------------------------------------------------------------- nibble packing
def pack_nibbles(code):
    """code [..., 2m] (values < 16) -> bytes [..., m]: element 2i low nibble, 2i+1 high."""
    c = code.astype(np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(b):
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0x0F
    out[..., 1::2] = b >> 4
    return out


def pack_bitplane(bits):
    """bits [..., 8m] (0/1) -> bytes [..., m]: bit j of byte k is element 8k + j."""
    b = bits.astype(np.uint8)
    out = np.zeros(b.shape[:-1] + (b.shape[-1] // 8,), dtype=np.uint8)
    for j in range(8):
        out |= (b[..., j::8] << j).astype(np.uint8)
    return out


def unpack_bitplane(b):
    out = np.empty(b.shape[:-1] + (8 * b.shape[-1],), dtype=np.uint8)
    for j in range(8):
        out[..., j::8] = (b >> j) & 1
    return out


def pack_crumbs(vals):
    """vals [..., 4m] (values < 4) -> bytes [..., m]: element 4k + j at bits 2j of byte k."""
    v = vals.astype(np.uint8)
    out = np.zeros(v.shape[:-1] + (v.shape[-1] // 4,), dtype=np.uint8)
    for j in range(4):
        out |= (v[..., j::4] << (2 * j)).astype(np.uint8)
    return out


def unpack_crumbs(b):
    out = np.empty(b.shape[:-1] + (4 * b.shape[-1],), dtype=np.uint8)
    for j in range(4):
        out[..., j::4] = (b >> (2 * j)) & 3
    return out
