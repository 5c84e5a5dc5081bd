"""Pins of the oracle's KVarN balancing and row rounding — CPU only.

SJ-KVaRN §2.2 (balancing of a 128 x 256 tile by alternating row/column passes until
spreads match; 16 passes; per-row b-bit rounding with its own scale and zero point; fp16
scales) and §3 (2,304 B of scales per record per KV head = 0.28125 bits per value).
The exact scales of a balanced tile are parity unpinned (no worked example on the pages);
these tests pin the invariants.
"""

import numpy as np
import pytest

from oracle import kvarn

RNG = np.random.default_rng(5)


def _tile(outliers=8, factor=16.0):
    x = RNG.standard_normal((128, 256)).astype(np.float32)
    ch = RNG.choice(256, outliers, replace=False)
    x[:, ch] *= factor
    return x


def test_final_column_spread_is_one_and_factorisation():
    X = _tile()
    Y, r, c = kvarn.balance(X)
    Y64 = Y.astype(np.float64)
    col_std = Y64.std(axis=0)
    assert np.max(np.abs(col_std - 1)) < 1e-5
    # rows balanced too after 16 passes (spreads similar)
    assert np.max(np.abs(Y64.std(axis=1) - 1)) < 0.05
    recon = r.astype(np.float64)[:, None] * Y64 * c.astype(np.float64)[None, :]
    assert np.max(np.abs(recon - X) / (np.abs(X) + 1e-3)) < 1e-4


def test_fixed_point_of_sign_tile():
    # X = alpha * a_t * b_j with balanced sign vectors: one row pass makes every row spread
    # exactly alpha (power of two: all sums exact), after which Y is the sign pattern with
    # unit spreads, so r = alpha, c = 1 exactly.
    alpha = np.float32(0.5)
    a = np.array([1, -1] * 64, np.float32)
    b = np.array([1, 1, -1, -1] * 64, np.float32)
    X = alpha * a[:, None] * b[None, :]
    Y, r, c = kvarn.balance(X)
    assert np.all(r == alpha) and np.all(c == 1) and np.array_equal(Y, a[:, None] * b[None, :])
    code, S, Z, C = kvarn.encode(X, 4)
    # lo = -1, hi = 1: S = fp16(0.5 * 2 / 15) = 0x2c44, Z = fp16(-0.5) = 0xb800, C = 1
    assert np.all(S.view(np.uint16) == 0x2C44) and np.all(Z.view(np.uint16) == 0xB800)
    assert np.all(C.view(np.uint16) == 0x3C00)
    assert np.array_equal(code, np.where(X > 0, 15, 0))
    assert np.allclose(kvarn.decode(code, S, Z, C), X, atol=0.5 * 15 * 2 ** -14 + 1e-3)


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_row_rounding_error_bound(bits):
    X = _tile()
    code, S, Z, C = kvarn.encode(X, bits)
    assert code.max() <= 2 ** bits - 1
    Xr = kvarn.decode(code, S, Z, C)
    S32, C32 = S.astype(np.float32)[:, None], C.astype(np.float32)[None, :]
    # half a step, plus the fp16 rounding of S, Z, C (relative 2^-11 each) over the row range
    bound = 0.5 * S32 * np.abs(C32) + 3 * 2 ** -11 * (np.abs(X) + (2 ** bits) * S32 * np.abs(C32))
    assert np.all(np.abs(Xr - X) <= bound + 1e-6)
    # the row min / max are reconstructed within that bound too (codes 0 and Q are used)
    assert np.all(code.min(axis=1) == 0) and np.all(code.max(axis=1) >= 2 ** bits - 2)


def test_tile_bytes_and_bits_per_value():
    X = _tile()
    for bits in (2, 3, 4, 5, 6, 8):
        code, S, Z, C = kvarn.encode(X, bits)
        for role in "KV":
            b = kvarn.pack_codes(code, bits, role)
            assert b.size == 4096 * bits
            assert np.array_equal(kvarn.unpack_codes(b, bits, role), code)
        sb = kvarn.scale_block(S, Z, C)
        assert sb.nbytes == 1152 and np.all(sb[512:] == 0)
    # SJ-KVaRN §3: 2,304 B of scales per record per head (K + V) adds 0.28125 bits/value
    assert 2 * 1152 * 8 / (2 * 128 * 256) == 0.28125
    assert (4096 * 4 + 1152) * 8 / (128 * 256) == 4.28125


def test_role_layouts():
    code = (np.arange(128 * 256) % 32).astype(np.uint8).reshape(128, 256)
    bK = kvarn.pack_codes(code, 5, "K")
    bV = kvarn.pack_codes(code, 5, "V")
    # K: token 1's first byte holds channels 0, 1 of token 1 (low nibbles of codes 0, 1)
    assert bK[128] == (code[1, 0] & 15) | ((code[1, 1] & 15) << 4)
    # V: channel 1's first byte holds tokens 0, 1 of channel 1
    assert bV[64] == (code[0, 1] & 15) | ((code[1, 1] & 15) << 4)
    # high planes: K row t occupies 32 B after the 16 KiB low plane; V row c 16 B
    assert bK[16384 + 32 * 2] & 1 == code[2, 0] >> 4
    assert (bV[16384 + 16 * 3] >> 2) & 1 == code[2, 3] >> 4


def test_plane_layouts_of_other_widths():
    """2-bit: four codes per byte, LSB first; 3-bit: that 2-bit plane, then a one-bit plane;
    6-bit: the nibble plane, then a 2-bit plane; 8-bit: one byte per code."""
    rng = np.random.default_rng(3)
    for bits in (2, 3, 6, 8):
        code = rng.integers(0, 2 ** bits, (128, 256)).astype(np.uint8)
        bK = kvarn.pack_codes(code, bits, "K")
        bV = kvarn.pack_codes(code, bits, "V")
        if bits in (2, 3):
            lo = code & 3
            assert bK[64 * 5 + 2] == lo[5, 8] | (lo[5, 9] << 2) | (lo[5, 10] << 4) | (lo[5, 11] << 6)
            assert bV[32 * 7 + 1] == lo[4, 7] | (lo[5, 7] << 2) | (lo[6, 7] << 4) | (lo[7, 7] << 6)
        if bits == 3:   # one-bit plane after the 8 KiB 2-bit plane: K rows of 32 B, V rows of 16 B
            assert (bK[8192 + 32 * 9 + 1] >> 3) & 1 == code[9, 11] >> 2
            assert (bV[8192 + 16 * 2 + 3] >> 5) & 1 == code[29, 2] >> 2
        if bits == 6:   # 2-bit plane after the 16 KiB nibble plane
            assert bK[128 * 3] == (code[3, 0] & 15) | ((code[3, 1] & 15) << 4)
            assert (bK[16384 + 64 * 3] >> 2) & 3 == code[3, 1] >> 4
        if bits == 8:
            assert np.array_equal(bK.reshape(128, 256), code) and np.array_equal(bV.reshape(256, 128), code.T)


def test_constant_rows_and_zero_tile():
    X = np.zeros((128, 256), np.float32)
    code, S, Z, C = kvarn.encode(X, 4)
    assert np.all(S == 0) and np.all(code == 0) and np.all(kvarn.decode(code, S, Z, C) == 0)


# ------------------------------------------------------------------ 8-pass keep-best balancing
# SJ-KVaRN §2.2: the KVarN reference configuration runs 8 passes and keeps the best scales
# seen. Reading (the format fixes it): a state is measured by the largest |sigma - 1| over the
# lines the last pass did not balance; the kept state is the smallest, the earliest on a tie.

def _alternating_tile(alpha):
    """32 rows of a balanced sign pattern (x alpha) over 96 zero rows: every sum is exact, the
    column spreads after a row pass are sqrt(32/128) = 0.5 and the row spreads after a column
    pass are 2, so the imbalance alternates 0.5, 1, 0.5, 1, ... exactly."""
    a = np.array([1, -1] * 16, np.float32)
    b = np.array([1, 1, -1, -1] * 64, np.float32)
    X = np.zeros((128, 256), np.float32)
    X[:32] = alpha * a[:, None] * b[None, :]
    return X, a, b


def test_best8_exact_alternation_keeps_the_first_pass():
    alpha = np.float32(0.25)
    X, a, b = _alternating_tile(alpha)
    Y, r, c, best, eps = kvarn.balance_best(X)
    assert eps.tolist() == [0.5, 1.0] * 4
    assert int(best) == 0                                   # ties: the earliest state
    assert np.all(r[:32] == alpha) and np.all(r[32:] == 1) and np.all(c == 1)
    assert np.array_equal(Y[:32], a[:, None] * b[None, :]) and not Y[32:].any()
    code, S, Z, C = kvarn.encode(X, 4, "best8")
    # rows 0..31: lo = -1, hi = 1: S = fp16(0.25 * 2 / 15), Z = fp16(-0.25); zero rows: S = Z = 0
    assert np.all(S[:32] == np.float16(np.float32(0.5) / np.float32(15))) and np.all(Z[:32] == np.float16(-0.25))
    assert not S[32:].view(np.uint16).any() and not Z[32:].view(np.uint16).any()
    assert np.all(C.view(np.uint16) == 0x3C00)
    assert np.array_equal(code[:32], np.where(X[:32] > 0, 15, 0)) and not code[32:].any()
    # the 16-pass rule keeps the last (column) pass instead: 8 column passes of 0.5, 7 row
    # passes of 2 after the first
    Yf, rf, cf = kvarn.balance(X)
    assert np.all(cf == 2.0 ** -8) and np.all(rf[:32] == alpha * 2 ** 7)


def _balance_fp64(X, passes=8):
    """Plain fp64 restatement of the passes and the imbalance measure (numpy std, no trees)."""
    Y = X.astype(np.float64)
    r, c = np.ones(128), np.ones(256)
    states, eps = [], []
    for p in range(passes):
        if p % 2 == 0:
            s = Y.std(axis=1)
            s = np.where(s <= 2.0 ** -20, 1.0, s)
            Y, r = Y / s[:, None], r * s
            o = Y.std(axis=0)
        else:
            s = Y.std(axis=0)
            s = np.where(s <= 2.0 ** -20, 1.0, s)
            Y, c = Y / s[None, :], c * s
            o = Y.std(axis=1)
        o = np.where(o <= 2.0 ** -20, 1.0, o)
        states.append((Y, r, c))
        eps.append(np.max(np.abs(o - 1)))
    return states, np.array(eps)


def _tiles():
    rng = np.random.default_rng(17)
    out = []
    for i in range(6):
        x = rng.standard_normal((128, 256)).astype(np.float32)
        x[:, rng.choice(256, 8, replace=False)] *= 16
        if i % 2 == 0:
            x[rng.choice(128, 3, replace=False)] = 0          # dead rows: no joint balance exists
        if i % 3 == 0:
            x *= np.exp(2 * rng.standard_normal((128, 1))).astype(np.float32)
        out.append(x)
    return out


def test_best8_matches_fp64_brute_force():
    seen_early = False
    for X in _tiles():
        Y, r, c, best, eps = kvarn.balance_best(X)
        states, eps64 = _balance_fp64(X)
        assert np.allclose(eps, eps64, rtol=1e-4, atol=1e-6)
        order = np.argsort(eps64, kind="stable")
        if eps64[order[1]] - eps64[order[0]] > 1e-4 * eps64[order[0]]:
            assert int(best) == int(order[0])
        b = int(best)
        assert eps[b] == eps.min() and b == int(np.flatnonzero(eps == eps.min())[0])
        Y64, r64, c64 = states[b]
        assert np.allclose(r, r64, rtol=1e-5) and np.allclose(c, c64, rtol=1e-5)
        assert np.allclose(Y, Y64, rtol=1e-4, atol=1e-5)
        # the kept state still factorises the tile
        recon = r.astype(np.float64)[:, None] * Y.astype(np.float64) * c.astype(np.float64)[None, :]
        assert np.max(np.abs(recon - X)) <= 1e-5 * np.max(np.abs(X))
        seen_early |= b < 7
    assert seen_early          # the dead-row tiles keep an earlier pass than the last


@pytest.mark.parametrize("bits", [2, 4, 5])
def test_best8_row_rounding_error_bound(bits):
    for X in _tiles()[:3]:
        code, S, Z, C = kvarn.encode(X, bits, "best8")
        Xr = kvarn.decode(code, S, Z, C)
        # every value within half a step of its row (times its column scale), plus the fp16
        # rounding of the scales
        step = np.abs(S.astype(np.float64))[:, None] * np.abs(C.astype(np.float64))[None, :]
        err = np.abs(Xr.astype(np.float64) - X)
        assert np.all(err <= 0.5 * step + 4e-3 * np.abs(X) + 1e-3 * step + 1e-6)
