"""The seal kernel reads the TBQ4 index #{k : u > beta_k} from a 2,048-bucket table indexed by
the top 11 bits of the fp32 value u (sign, exponent, two mantissa bits), as base + (u > thr).
That is exact only if no bucket holds two boundaries. These CPU tests check the property on
the oracle's boundary table and compare the bucket rule with the plain count (the TBQ4
definition of the page "KV cache math", section "Worked example"), including the values
that sit on a boundary or next to one.
"""

import numpy as np

from oracle import tables


def bucket_table(bnd):
    """(thr, base) per bucket, the same rule the kernel builds in shared memory."""
    thr = np.full(2048, np.inf, dtype=np.float32)
    base = np.zeros(2048, dtype=np.int64)
    count = np.zeros(2048, dtype=np.int64)
    for k in range(2048):
        lo = np.uint32(k << 21)
        hi = np.uint32(lo | 0x1FFFFF)
        if ((int(lo) >> 23) & 0xFF) == 0xFF:          # infinities and NaNs: index 0
            continue
        neg = bool(int(lo) >> 31)
        vmin = np.array([hi if neg else lo], dtype=np.uint32).view(np.float32)[0]
        vmax = np.array([lo if neg else hi], dtype=np.uint32).view(np.float32)[0]
        for b in bnd:
            if b < vmin:
                base[k] += 1
            elif b <= vmax:
                thr[k] = b
                count[k] += 1
    return thr, base, count


def lookup(u, thr, base):
    bk = (u.view(np.uint32) >> np.uint32(21)).astype(np.int64)
    return base[bk] + (u > thr[bk]).astype(np.int64)


def plain_index(u, bnd):
    return (u[:, None] > bnd[None, :]).sum(axis=1)


def test_every_bucket_holds_at_most_one_boundary():
    _, bnd = tables.tbq4_tables()
    thr, base, count = bucket_table(bnd)
    assert count.max() == 1
    assert count.sum() == 15 + 1          # beta_8 = 0 sits in the buckets of +0 and of -0
    # consecutive positive boundaries differ by more than a bucket's span (ratio 1.25)
    pos = bnd[bnd > 0].astype(np.float64)
    assert np.min(pos[1:] / pos[:-1]) > 1.25


def test_bucket_rule_equals_the_count():
    _, bnd = tables.tbq4_tables()
    thr, base, _ = bucket_table(bnd)
    rng = np.random.default_rng(5)
    sigma = np.float32(1 / np.sqrt(128))
    u = (rng.standard_normal(400_000) * sigma).astype(np.float32)
    # boundaries, their neighbours one ulp away on both sides, zeros and the unit extremes
    edge = np.concatenate([bnd, np.nextafter(bnd, np.float32(np.inf)), np.nextafter(bnd, np.float32(-np.inf)),
                           np.array([0.0, -0.0, 1.0005, -1.0005, 1e-30, -1e-30], dtype=np.float32)])
    u = np.concatenate([u, edge.astype(np.float32)])
    assert np.array_equal(lookup(u, thr, base), plain_index(u, bnd))


def test_nan_gives_index_zero():
    _, bnd = tables.tbq4_tables()
    thr, base, _ = bucket_table(bnd)
    u = np.array([np.nan, -np.nan], dtype=np.float32)
    assert np.array_equal(lookup(u, thr, base), plain_index(u, bnd))
