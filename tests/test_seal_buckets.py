"""The seal kernel reads the TBQ4 index #{k : u > beta_k} from a 2,048-bucket table as the top
four bits of entry + key. Over an order-preserving integer key of the fp32 value u (its bits,
with the magnitude bits inverted for negative values) a bucket is the key's top 11 bits, and
the entry holds base << 28 and a bias that makes the low 28 bits carry exactly when u exceeds
the bucket's boundary. That is exact only if no bucket holds two boundaries. The kernel indexes
the table by u's own top 11 bits and adds the absolute value of u's bits as a 32-bit integer
(2^32 minus the bits for negative values: the order-preserving key plus 2^31 + 1), so it stores
a negative bucket's entry at the index of its bits' bucket, raised by 2^31 - 1. These CPU tests check the property on the oracle's boundary
table and compare the kernel's rule, built here the way the kernel builds it, with the plain
count (the TBQ4 definition of the page "KV cache math", section "Worked example"), including
the values that sit on a boundary or next to one, both zeros and NaNs.
"""

import numpy as np
import pytest

from oracle import tables


def fkey(u):
    """Order-preserving key of fp32 values (uint64 arithmetic on the 32-bit patterns)."""
    b = np.asarray(u, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return b ^ np.where(b >> np.uint64(31), np.uint64(0x7FFFFFFF), np.uint64(0))


def bucket_table(bnd):
    """(entry, base, count) per key bucket (entry over the order-preserving key)."""
    entry = np.zeros(2048, dtype=np.uint64)
    base = np.zeros(2048, dtype=np.int64)
    count = np.zeros(2048, dtype=np.int64)
    for k in range(2048):
        klo = k << 21
        khi = klo | 0x1FFFFF
        neg = k >= 1024
        flip = 0x7FFFFFFF if neg else 0
        blo, bhi = klo ^ flip, khi ^ flip
        t = 0x1FFFFF
        if ((blo >> 23) & 0xFF) != 0xFF:               # infinities and NaNs: index 0
            vmin = np.array([blo], dtype=np.uint32).view(np.float32)[0]
            vmax = np.array([bhi], dtype=np.uint32).view(np.float32)[0]
            for b in bnd:
                if b < vmin:
                    base[k] += 1
                elif b <= vmax:
                    t = 0x1FFFFF if (neg and b == 0) else int(fkey(b)) & 0x1FFFFF
                    count[k] += 1
        entry[k] = ((int(base[k]) << 28) + (0x0FFFFFFF - t) - klo) % (1 << 32)
    return entry, base, count


def kernel_table(entry):
    """The table as the kernel stores it: indexed by the bits' bucket, negative entries + 2^31 - 1."""
    qt = np.zeros(2048, dtype=np.uint64)
    for k in range(2048):
        if k >= 1024:
            qt[k ^ 0x3FF] = (int(entry[k]) + (1 << 31) - 1) % (1 << 32)
        else:
            qt[k] = entry[k]
    return qt


def lookup(u, entry):
    """The kernel's rule: table at u's bits' top 11 bits, plus |bits| as a 32-bit integer."""
    qt = kernel_table(entry)
    b = np.asarray(u, dtype=np.float32).view(np.uint32).astype(np.uint64)
    key = np.where(b >> np.uint64(31), (np.uint64(1 << 32) - b) % np.uint64(1 << 32), b)
    return (((qt[(b >> np.uint64(21)).astype(np.int64)] + key) % np.uint64(1 << 32)) >> np.uint64(28)).astype(np.int64)


def lookup_key(u, entry):
    """The same index over the order-preserving key directly."""
    key = fkey(u)
    return (((entry[(key >> np.uint64(21)).astype(np.int64)] + key) % np.uint64(1 << 32)) >> np.uint64(28)).astype(np.int64)


def plain_index(u, bnd):
    return (u[:, None] > bnd[None, :]).sum(axis=1)


def test_every_bucket_holds_at_most_one_boundary():
    _, bnd = tables.tbq4_tables()
    _, base, count = bucket_table(bnd)
    assert count.max() == 1
    assert count.sum() == 15 + 1          # beta_8 = 0 sits in the buckets of +0 and of -0
    # consecutive positive boundaries differ by more than a bucket's span (ratio 1.25)
    pos = bnd[bnd > 0].astype(np.float64)
    assert np.min(pos[1:] / pos[:-1]) > 1.25


@pytest.mark.parametrize("table", ["tbq4", "turbo3"])
def test_bucket_rule_equals_the_count(table):
    _, bnd = (tables.tbq4_tables if table == "tbq4" else tables.tbq3_tables)()
    entry, _, count = bucket_table(bnd)
    assert count.max() == 1
    rng = np.random.default_rng(5)
    sigma = np.float32(1 / np.sqrt(128))
    u = (rng.standard_normal(400_000) * sigma).astype(np.float32)
    # boundaries, their neighbours one ulp away on both sides, zeros and the unit extremes
    edge = np.concatenate([bnd, np.nextafter(bnd, np.float32(np.inf)), np.nextafter(bnd, np.float32(-np.inf)),
                           np.array([0.0, -0.0, 1.0005, -1.0005, 1e-30, -1e-30], dtype=np.float32)])
    u = np.concatenate([u, edge.astype(np.float32)])
    assert np.array_equal(lookup(u, entry), plain_index(u, bnd))
    assert np.array_equal(lookup_key(u, entry), plain_index(u, bnd))


@pytest.mark.parametrize("table", ["tbq4", "turbo3"])
def test_kernel_rule_equals_key_rule_at_every_bucket_edge(table):
    """Both rules at the first and last two bit patterns of every bucket and next to every
    boundary's pattern: equal sums mod 2^32 wherever the index is defined."""
    _, bnd = (tables.tbq4_tables if table == "tbq4" else tables.tbq3_tables)()
    entry, _, _ = bucket_table(bnd)
    k = np.arange(2048, dtype=np.uint64) << np.uint64(21)
    pats = np.concatenate([k, k + 1, k + 0x1FFFFE, k + 0x1FFFFF])
    bb = np.asarray(bnd, dtype=np.float32).view(np.uint32).astype(np.int64)
    near = np.concatenate([bb + d for d in (-1, 0, 1)] + [(bb ^ (1 << 31)) + d for d in (-1, 0, 1)])
    pats = np.concatenate([pats, (near % (1 << 32)).astype(np.uint64)]).astype(np.uint32)
    u = pats.view(np.float32)
    assert np.array_equal(lookup(u, entry), lookup_key(u, entry))


def test_nan_gives_index_zero():
    _, bnd = tables.tbq4_tables()
    entry, _, _ = bucket_table(bnd)
    u = np.array([np.nan, -np.nan], dtype=np.float32)
    assert np.array_equal(lookup(u, entry), plain_index(u, bnd))
