"""Pins of the oracle's rotations — CPU only.

SJ-KVaRN §2.2: 256-point Hadamard, orthonormal, queries rotated the same way so q.k is
unchanged; KV cache math "rotate first": sign flip, WHT, sign flip; q.k = (Hq).(Hk).
"""

import numpy as np
import pytest
from scipy.linalg import hadamard

from oracle import rotation, tables

RNG = np.random.default_rng(7)


@pytest.mark.parametrize("n", [2, 4, 8, 16, 32, 64, 128, 256])
def test_fwht_equals_sylvester_matrix(n):
    x = RNG.standard_normal((5, n))
    assert np.allclose(rotation.fwht(x), x @ hadamard(n).T, atol=1e-12)


def test_had256_fp32_against_matrix_and_orthonormal():
    x = RNG.standard_normal((7, 512)).astype(np.float32)
    y = rotation.rotate(x, rotation.HAD256)
    H = hadamard(256) / 16.0
    ref = np.concatenate([x[:, :256].astype(np.float64) @ H.T, x[:, 256:].astype(np.float64) @ H.T], axis=1)
    assert np.max(np.abs(y - ref)) < 1e-5 * np.max(np.abs(ref))
    assert np.allclose(H @ H.T, np.eye(256))
    # rotation is an involution up to rounding: H/16 applied twice is the identity
    assert np.allclose(rotation.rotate(y, rotation.HAD256), x, atol=1e-5)


def test_tbq128_against_matrix_and_inverse():
    s1, s2 = tables.tbq_signs()
    x = RNG.standard_normal((3, 256))
    R = np.diag(s2.astype(np.float64)) @ hadamard(128) @ np.diag(s1.astype(np.float64)) / np.sqrt(128)
    ref = np.concatenate([x[:, :128] @ R.T, x[:, 128:] @ R.T], axis=1)
    assert np.allclose(rotation.rotate_f64(x, rotation.TBQ128), ref, atol=1e-12)
    assert np.allclose(R @ R.T, np.eye(128), atol=1e-12)
    back = rotation.rotate_f64(rotation.rotate_f64(x, rotation.TBQ128), rotation.TBQ128, inverse=True)
    assert np.allclose(back, x, atol=1e-12)
    y32 = rotation.rotate(x.astype(np.float32), rotation.TBQ128)
    assert np.max(np.abs(y32 - ref)) < 1e-5


@pytest.mark.parametrize("kind", [rotation.HAD256, rotation.TBQ128])
def test_dot_products_survive_rotation(kind):
    q = RNG.standard_normal((4, 512))
    k = RNG.standard_normal((9, 512))
    rq, rk = rotation.rotate_f64(q, kind), rotation.rotate_f64(k, kind)
    assert np.allclose(rq @ rk.T, q @ k.T, atol=1e-12)
    q32, k32 = q.astype(np.float32), k.astype(np.float32)
    d32 = rotation.rotate(q32, kind).astype(np.float64) @ rotation.rotate(k32, kind).astype(np.float64).T
    assert np.max(np.abs(d32 - q32.astype(np.float64) @ k32.astype(np.float64).T)) < 1e-4


def test_outlier_energy_is_spread():
    # SJ-KVaRN §2.2: rotation spreads an outlier's energy across all channels.
    x = np.zeros(256, np.float32)
    x[17] = 100.0
    y = rotation.rotate(x, rotation.HAD256)
    assert np.allclose(np.abs(y), 100.0 / 16)
