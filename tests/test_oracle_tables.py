"""Pins of the oracle's format constants (sign words, Lloyd-Max table) — CPU only."""

import math

import numpy as np
from scipy import integrate

from oracle import tables


def test_splitmix64_published_vector():
    # Reference outputs of splitmix64 seeded with 1234567 (Vigna's public test vector).
    assert tables.splitmix64(1234567, 5) == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]


def test_sign_expansion_bits():
    s1, s2 = tables.tbq_signs()
    w = tables.sign_words()
    assert s1.shape == (128,) and s2.shape == (128,)
    assert set(np.unique(s1)) <= {-1.0, 1.0}
    # bit i of word 0 set <=> s1[i] == -1; bit 3 of word 3 set <=> s2[64+3] == -1
    for i in range(64):
        assert (s1[i] < 0) == bool((w[0] >> i) & 1)
        assert (s2[64 + i] < 0) == bool((w[3] >> i) & 1)
    # both vectors are far from constant (a seed mistake would typically give +1 everywhere)
    assert 40 < int((s1 < 0).sum()) < 90 and 40 < int((s2 < 0).sum()) < 90


def test_lloyd_two_level_closed_form():
    # 1-bit Lloyd-Max for N(0,1): +-E|X| = +-sqrt(2/pi)
    c = tables.lloyd_max_gaussian(2, iters=200)
    assert abs(c[1] - math.sqrt(2 / math.pi)) < 1e-15 and c[0] == -c[1]


def test_lloyd_16_matches_max_1960_table():
    # J. Max, "Quantizing for minimum distortion" (1960), 16-level Gaussian output levels.
    printed = [0.1284, 0.3881, 0.6568, 0.9424, 1.2562, 1.6180, 2.0690, 2.7326]
    c = tables.lloyd_max_gaussian(16)
    assert all(abs(a - b) < 6e-5 for a, b in zip(c[8:], printed))
    assert all(c[15 - j] == -c[j] for j in range(16))


def test_lloyd_16_centroid_condition_by_quadrature():
    # Independent check: each level is the conditional mean of its cell (numerical quadrature).
    c = tables.lloyd_max_gaussian(16)
    b = [-math.inf] + [(c[k - 1] + c[k]) / 2 for k in range(1, 16)] + [math.inf]
    phi = lambda x: math.exp(-x * x / 2) / math.sqrt(2 * math.pi)
    for k in range(16):
        mass = integrate.quad(phi, b[k], b[k + 1], epsabs=1e-15, epsrel=1e-13)[0]
        mean = integrate.quad(lambda x: x * phi(x), b[k], b[k + 1], epsabs=1e-15, epsrel=1e-13)[0] / mass
        assert abs(mean - c[k]) < 1e-9


def test_tbq4_fp32_tables():
    cent, bnd = tables.tbq4_tables()
    sigma = 1 / math.sqrt(128)
    c = tables.lloyd_max_gaussian(16)
    assert cent.dtype == np.float32 and bnd.dtype == np.float32
    assert np.all(np.diff(cent) > 0) and np.all(np.diff(bnd) > 0)
    assert bnd[7] == 0.0
    for j in range(16):
        assert cent[j] == np.float32(sigma * c[j])
    for k in range(1, 16):
        assert cent[k - 1] < bnd[k - 1] < cent[k]
