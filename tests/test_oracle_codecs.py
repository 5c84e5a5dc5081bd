"""Pins of the oracle's block codecs (tq6_0, TBQ4, Q8_0, Q4_0) — CPU only."""

import json
import math
import os

import numpy as np
import pytest

from oracle import codecs, tables

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "block_codecs.json")))
RNG = np.random.default_rng(11)


def _block(case):
    x = np.zeros(case["n"], np.float32)
    for i, v in case["x_nonzero"].items():
        x[int(i)] = v
    return x


def _hex(a):
    return [format(int(b), "02x") for b in np.asarray(a).reshape(-1)]


# ------------------------------------------------------------------ hand-derived blocks
def test_tq6_golden_block():
    g = GOLD["tq6_0"]
    d, code = codecs.tq6_encode(_block(g))
    assert format(int(d.view(np.uint16)[0]), "04x") == g["d_bits"]
    assert list(code[0, :8]) == g["codes_head"] and np.all(code[0, 8:] == g["code_rest"])
    ql, qh = codecs.tq6_pack(code[0])
    assert _hex(ql[:4]) == g["ql_head"] and set(_hex(ql[4:])) == {g["ql_rest"]}
    assert _hex(qh[:2]) == g["qh_head"] and set(_hex(qh[2:])) == {g["qh_rest"]}
    assert ql.size + qh.size + 2 == 98


def test_q8_golden_block():
    g = GOLD["q8_0"]
    d, q = codecs.q8_encode(_block(g))
    assert format(int(d.view(np.uint16)[0]), "04x") == g["d_bits"]
    assert list(q[0, :5]) == g["q_head"] and np.all(q[0, 5:] == 0)
    assert _hex(q[0, :5].view(np.uint8)) == g["bytes_head"]
    assert q.size + 2 == 34


def test_q4_golden_block():
    g = GOLD["q4_0"]
    d, c = codecs.q4_encode(_block(g))
    assert format(int(d.view(np.uint16)[0]), "04x") == g["d_bits"]
    assert list(c[0, :5]) == g["codes_head"] and np.all(c[0, 5:] == g["code_rest"])
    b = codecs.pack_nibbles(c[0])
    assert _hex(b[:3]) == g["bytes_head"] and set(_hex(b[3:])) == {g["byte_rest"]}
    assert b.size + 2 == 18


def test_tbq4_golden_blocks():
    g = GOLD["tbq4"]
    y = np.zeros(128, np.float32)
    y[0] = 1.0
    n16, idx = codecs.tbq4_encode(y)
    assert format(int(n16.view(np.uint16)[0]), "04x") == g["one_hot"]["n_bits"]
    assert idx[0, 0] == g["one_hot"]["idx_head"] and np.all(idx[0, 1:] == g["one_hot"]["idx_rest"])
    b = codecs.pack_nibbles(idx[0])
    assert _hex(b[:1]) == [g["one_hot"]["byte_head"]] and set(_hex(b[1:])) == {g["one_hot"]["byte_rest"]}
    assert b.size + 2 == 66
    y = np.full(128, 1 / 16, np.float32)
    n16, idx = codecs.tbq4_encode(y)
    assert format(int(n16.view(np.uint16)[0]), "04x") == g["const_1_16"]["n_bits"]
    assert np.all(idx == g["const_1_16"]["idx"])
    assert set(_hex(codecs.pack_nibbles(idx[0]))) == {g["const_1_16"]["byte"]}


# ------------------------------------------------------------------ packing (bit-exact layout)
def test_tq6_pack_exhaustive_positions_and_values():
    # KV cache math reports a 3-bit packing bug that corrupted values 3-7 of each group:
    # every code value at every position must round-trip, with the stated bit positions.
    for v in range(64):
        for pos in range(128):
            code = np.full(128, 32, np.uint8)
            code[pos] = v
            ql, qh = codecs.tq6_pack(code)
            assert (ql[pos // 2] >> (4 * (pos % 2))) & 0xF == v & 0xF
            assert (qh[pos // 4] >> (2 * (pos % 4))) & 0x3 == v >> 4
            assert np.array_equal(codecs.tq6_unpack(ql, qh), code)


def test_nibble_and_bitplane_exhaustive():
    for v in range(16):
        for pos in range(32):
            c = np.zeros(32, np.uint8)
            c[pos] = v
            b = codecs.pack_nibbles(c)
            assert (b[pos // 2] >> (4 * (pos % 2))) & 0xF == v
            assert np.array_equal(codecs.unpack_nibbles(b), c)
    for pos in range(64):
        bits = np.zeros(64, np.uint8)
        bits[pos] = 1
        b = codecs.pack_bitplane(bits)
        assert b[pos // 8] == 1 << (pos % 8) and b.sum() == b[pos // 8]
        assert np.array_equal(codecs.unpack_bitplane(b), bits)


# ------------------------------------------------------------------ error bounds and invariants
def _fp16_err(d):
    return d.astype(np.float32) * np.float32(2 ** -11)


@pytest.mark.parametrize("scale", [1e-3, 1.0, 40.0])
def test_tq6_error_bound_and_idempotence(scale):
    x = (RNG.standard_normal((64, 256)) * scale).astype(np.float32)
    d, code = codecs.tq6_encode(x)
    xr = codecs.tq6_decode(d, code)
    half = np.repeat(d.astype(np.float32) / 2, 128, axis=-1) * (1 + 1e-6)
    # the stored scale may round below absmax/31, letting the extreme clip by < 31 * ulp(d)
    slack = np.repeat(31 * _fp16_err(d), 128, axis=-1)
    assert np.all(np.abs(x - xr) <= half + slack)
    d2, code2 = codecs.tq6_encode(xr)
    assert np.array_equal(code2, code)
    assert np.all((code >= 1) & (code <= 63))


def test_zero_blocks():
    d, c = codecs.tq6_encode(np.zeros(128, np.float32))
    assert d[0] == 0 and np.all(c == 32)
    n, i = codecs.tbq4_encode(np.zeros(128, np.float32))
    assert n[0] == 0 and np.all(codecs.tbq4_decode(n, i) == 0)
    d, q = codecs.q8_encode(np.zeros(32, np.float32))
    assert d[0] == 0 and np.all(q == 0)
    d, c = codecs.q4_encode(np.zeros(32, np.float32))
    assert d[0] == 0 and np.all(c == 8)


@pytest.mark.parametrize("enc,dec,qmax", [(codecs.q8_encode, codecs.q8_decode, 127),
                                          (codecs.q4_encode, codecs.q4_decode, 7)])
def test_q_block_error_bound_and_idempotence(enc, dec, qmax):
    x = (RNG.standard_normal((50, 128)) * 3).astype(np.float32)
    d, c = enc(x)
    xr = dec(d, c)
    half = np.repeat(d.astype(np.float32) / 2, 32, axis=-1) * (1 + 1e-6)
    slack = np.repeat(qmax * _fp16_err(d), 32, axis=-1)
    assert np.all(np.abs(x - xr) <= half + slack)
    d2, c2 = enc(xr)
    assert np.array_equal(c2, c)


def test_tbq4_index_is_nearest_centroid_and_mse():
    cent, bnd = tables.tbq4_tables()
    y = RNG.standard_normal((2000, 128)).astype(np.float32)
    n16, idx = codecs.tbq4_encode(y)
    u = y * (np.float32(1) / n16.astype(np.float32))
    # brute force over the 16 levels in fp64 (boundaries are midpoints -> nearest level)
    nearest = np.argmin(np.abs(u[..., None].astype(np.float64) - cent.astype(np.float64)), axis=-1)
    agree = np.mean(nearest.reshape(idx.shape) == idx)
    assert agree > 0.99999
    # distortion of unit-variance-per-block data ~ Lloyd-Max 16-level MSE (~0.0095 sigma^2)
    yr = codecs.tbq4_decode(n16, idx)
    rel_mse = np.mean((y - yr) ** 2) / np.mean(y ** 2)
    assert 0.0085 < rel_mse < 0.0110
    assert np.allclose(n16.astype(np.float64), np.linalg.norm(y.reshape(-1, 128), axis=1).reshape(n16.shape),
                       rtol=1e-3)


def test_tbq4_ties_go_low():
    # u exactly on boundary beta_9 (= bnd[8] = 0.0228) must take the lower cell, index 8.
    cent, bnd = tables.tbq4_tables()
    y = np.zeros(128, np.float32)
    y[0] = 1.0
    y[1] = bnd[8]
    n16, idx = codecs.tbq4_encode(y)
    assert n16[0] == 1.0            # sqrt(1 + 0.00052) rounds to fp16 1.0
    assert idx[0, 1] == 8 and idx[0, 0] == 15
    y[1] = np.nextafter(bnd[8], np.float32(1))
    assert codecs.tbq4_encode(y)[1][0, 1] == 9


# ----------------------------------------------------------------------------- Q5_0 / Q6_0 / Q4_1 / Q5_1
@pytest.mark.parametrize("L", [15, 31])
def test_qsym_error_bound_zero_and_grid(L):
    x = (RNG.standard_normal((400, 32)) * RNG.uniform(0.01, 50, (400, 1))).astype(np.float32)
    d, code = codecs.qsym_encode(x, L)
    xr = codecs.qsym_decode(d, code, L)
    d32 = d.astype(np.float32)          # [400, 1]: one block per row
    assert code.min() >= 1 and code.max() <= 2 * L + 1
    # half a step, plus the fp16 rounding of d over the block's range (|x| <= L d (1 + 2^-11))
    assert np.all(np.abs(xr.reshape(x.shape) - x) <= 0.5 * d32 + L * d32 * 2 ** -10)
    # the largest magnitude of each block is coded at level +-L (or next to it)
    assert np.all(np.abs(code.astype(int) - (L + 1)).max(axis=-1) >= L - 1)
    # values on the grid come back exactly, and their codes are stable
    d2, c2 = codecs.qsym_encode(xr, L)
    assert np.array_equal(codecs.qsym_decode(d2, c2, L), xr)
    # a zero block: d = 0 and every code the zero level L + 1
    dz, cz = codecs.qsym_encode(np.zeros(32, np.float32), L)
    assert dz[0] == 0 and np.all(cz == L + 1)


@pytest.mark.parametrize("Q", [15, 31])
def test_qmin_error_bound_extremes_and_constants(Q):
    x = (RNG.standard_normal((400, 32)) * RNG.uniform(0.01, 50, (400, 1)) + RNG.uniform(-5, 5, (400, 1))).astype(np.float32)
    d, m, code = codecs.qmin_encode(x, Q)
    xr = codecs.qmin_decode(d, m, code).reshape(x.shape)
    d32, m32 = d.astype(np.float32), m.astype(np.float32)      # [400, 1]: one block per row
    assert code.max() <= Q
    # half a step, plus the fp16 roundings of m and d (relative 2^-11) over the block's values
    bound = 0.5 * d32 + 2 ** -11 * np.abs(m32) + Q * d32 * 2 ** -10 + 1e-6
    assert np.all(np.abs(xr - x) <= bound)
    # the block's minimum takes code 0 and its maximum code Q (or next to them)
    lo = np.argmin(x, axis=-1)
    hi = np.argmax(x, axis=-1)
    assert np.all(code[np.arange(400), 0, lo] <= 1) and np.all(code[np.arange(400), 0, hi] >= Q - 1)
    # a constant block: d = 0, every code 0, decoded as fp16(c)
    dc, mc, cc = codecs.qmin_encode(np.full(32, 0.3, np.float32), Q)
    assert dc[0] == 0 and np.all(cc == 0)
    assert np.all(codecs.qmin_decode(dc, mc, cc) == np.float32(np.float16(0.3)))


def test_block_format_sizes_are_the_pages():
    """Packed record sizes per 32 values: q5_0 22 B, q6_0 26 B, q4_1 20 B, q5_1 24 B (the pages'
    block sizes, also in the oracle's byte table)."""
    from oracle.cache import encode_body, pack_body
    from oracle import sizes
    X = RNG.standard_normal((128, 256)).astype(np.float32)
    for fmt, b in (("q5_0", 22), ("q6_0", 26), ("q4_1", 20), ("q5_1", 24)):
        rec = encode_body(X, fmt)
        for role in "KV":
            assert pack_body(rec, fmt, role).size == 128 * 256 // 32 * b
        assert sizes.record_bytes(fmt, 256) == 128 * 256 // 32 * b


def test_crumb_packing_exhaustive():
    v = np.array([[a, b, c, d] for a in range(4) for b in range(4) for c in range(4) for d in range(4)], np.uint8)
    p = codecs.pack_crumbs(v)
    assert np.array_equal(p[:, 0], v[:, 0] | (v[:, 1] << 2) | (v[:, 2] << 4) | (v[:, 3] << 6))
    assert np.array_equal(codecs.unpack_crumbs(p), v)


# ----------------------------------------------------------------------------- turbo3 / tq5_0
def test_eight_level_lloyd_max_table():
    """turbo3's table: the 8-level Lloyd-Max quantizer of N(0,1) (Max 1960, Table I: levels
    +-0.2451, +-0.7560, +-1.3440, +-2.1520, distortion 0.03454), scaled by 1/sqrt(128)."""
    cent, bnd = tables.tbq3_tables()
    C = np.array(tables.lloyd_max_gaussian(8))
    assert np.allclose(C[4:], [0.2451, 0.7560, 1.3440, 2.1520], atol=1e-4)
    assert np.array_equal(cent[:4], -cent[:3:-1]) and bnd[3] == 0
    # each level is the conditional mean of its cell, boundaries the midpoints (fp64)
    b = [0.0] + [(C[4 + k - 1] + C[4 + k]) / 2 for k in range(1, 4)] + [math.inf]
    phi = lambda x: 0.0 if x == math.inf else math.exp(-x * x / 2) / math.sqrt(2 * math.pi)
    tail = lambda x: 0.0 if x == math.inf else 0.5 * math.erfc(x / math.sqrt(2))
    for k in range(4):
        assert abs((phi(b[k]) - phi(b[k + 1])) / (tail(b[k]) - tail(b[k + 1])) - C[4 + k]) < 1e-12
    # distortion E[(x - Q(x))^2] for N(0,1): 1 - sum_k P_k C_k^2 for the optimal quantizer
    mse = 1 - 2 * sum((tail(b[k]) - tail(b[k + 1])) * C[4 + k] ** 2 for k in range(4))
    assert abs(mse - 0.03454) < 1e-4


def test_turbo3_nearest_centroid_and_distortion():
    cent, bnd = tables.tbq3_tables()
    y = RNG.standard_normal((2000, 128)).astype(np.float32)
    n16, idx = codecs.turbo3_encode(y)
    assert idx.max() <= 7
    u = y * (np.float32(1) / n16.astype(np.float32))
    nearest = np.argmin(np.abs(u[..., None].astype(np.float64) - cent.astype(np.float64)), axis=-1)
    assert np.mean(nearest.reshape(idx.shape) == idx) > 0.99999
    rel_mse = np.mean((y - codecs.turbo3_decode(n16, idx)) ** 2) / np.mean(y ** 2)
    assert 0.031 < rel_mse < 0.038
    # a zero block: norm 0, u = 0 exceeds the three negative boundaries only (the boundary at 0
    # is a tie, which goes to the lower level): index 3
    z16, zi = codecs.turbo3_encode(np.zeros(128, np.float32))
    assert z16[0] == 0 and np.all(zi == 3)


def test_tq5_error_bound_zero_and_grid():
    x = (RNG.standard_normal((300, 128)) * RNG.uniform(0.01, 40, (300, 1))).astype(np.float32)
    d, code = codecs.tq5_encode(x)
    xr = codecs.tq5_decode(d, code).reshape(x.shape)
    d32 = d.astype(np.float32)
    assert code.min() >= 1 and code.max() <= 31
    assert np.all(np.abs(xr - x) <= 0.5 * d32 + 15 * d32 * 2 ** -10)
    d2, c2 = codecs.tq5_encode(xr)
    assert np.array_equal(codecs.tq5_decode(d2, c2), xr)
    dz, cz = codecs.tq5_encode(np.zeros(128, np.float32))
    assert dz[0] == 0 and np.all(cz == 16)


def test_rotated_comparator_sizes_are_the_pages():
    """turbo3 50 B and tq5_0 82 B per 128 values (KV cache math table; SJ-KVaRN §4.1)."""
    from oracle.cache import encode_body, pack_body
    from oracle import sizes
    X = RNG.standard_normal((128, 256)).astype(np.float32)
    for fmt, b in (("turbo3", 50), ("tq5_0", 82)):
        rec = encode_body(X, fmt)
        for role in "KV":
            assert pack_body(rec, fmt, role).size == 256 * b
        assert sizes.record_bytes(fmt, 256) == 256 * b
