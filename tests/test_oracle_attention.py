"""Pins of the oracle's decode attention (fp64) — CPU only.

KV Cache Precision Tail §2: regions' attention results combine under one softmax;
KV cache math "rotate first": q.k = (Hq).(Hk), the output is rotated back once.
"""

import numpy as np
import pytest
from scipy.special import softmax

from oracle import attention, rotation

RNG = np.random.default_rng(3)


def _regions(G=4, D=128, sizes=(7, 30, 1, 12)):
    doms = ["exact", "rot", "rot", "exact"]
    return [(d, RNG.standard_normal((n, D)), RNG.standard_normal((n, D))) for d, n in zip(doms, sizes)]


def test_single_region_matches_library_softmax():
    q = RNG.standard_normal((3, 128))
    K, V = RNG.standard_normal((50, 128)), RNG.standard_normal((50, 128))
    o = attention.attend(q, [("exact", K, V)], rotation.NONE, 0.3)
    assert np.allclose(o, softmax(0.3 * q @ K.T, axis=1) @ V, atol=1e-13)


@pytest.mark.parametrize("kind", [rotation.NONE, rotation.HAD256, rotation.TBQ128])
def test_rotated_regions_equal_unrotated_attention(kind):
    # Storing R k and R v and reading them with R q, then rotating the output back, must give
    # plain attention over k and v (orthonormal R). A dropped inverse or a wrong sign fails.
    D = 256
    q = RNG.standard_normal((6, D))
    K, V = RNG.standard_normal((40, D)), RNG.standard_normal((40, D))
    plain = softmax(0.1 * q @ K.T, axis=1) @ V
    Kr, Vr = rotation.rotate_f64(K, kind), rotation.rotate_f64(V, kind)
    regs = [("exact", K[:10], V[:10]), ("rot", Kr[10:33], Vr[10:33]), ("exact", K[33:], V[33:])]
    assert np.allclose(attention.attend(q, regs, kind, 0.1), plain, atol=1e-12)


@pytest.mark.parametrize("kind", [rotation.NONE, rotation.HAD256])
def test_lse_merge_equals_single_softmax(kind):
    q = RNG.standard_normal((4, 256))
    regs = _regions(D=256)
    a = attention.attend(q, regs, kind, 0.2)
    b = attention.lse_merge(attention.region_partials(q, regs, kind, 0.2), kind)
    assert np.max(np.abs(a - b)) < 1e-14 * max(1.0, np.max(np.abs(a)))
    # chunking one region further does not change the result
    split = []
    for d, K, V in regs:
        split += [(d, K[:len(K) // 2], V[:len(V) // 2]), (d, K[len(K) // 2:], V[len(V) // 2:])]
    c = attention.lse_merge(attention.region_partials(q, split, kind, 0.2), kind)
    assert np.max(np.abs(a - c)) < 1e-14 * max(1.0, np.max(np.abs(a)))


def test_special_cases():
    D = 128
    q = RNG.standard_normal((2, D))
    k = RNG.standard_normal(D)
    V = RNG.standard_normal((20, D))
    K = np.tile(k, (20, 1))
    # all keys equal -> uniform weights -> mean of V
    assert np.allclose(attention.attend(q, [("exact", K, V)], rotation.NONE, 1.0), np.tile(V.mean(0), (2, 1)))
    # one dominant score -> that V
    K2 = np.zeros((20, D))
    K2[13] = 1e3 * q[0]
    o = attention.attend(q[:1], [("exact", K2, V)], rotation.NONE, 1.0)
    assert np.allclose(o[0], V[13])


def test_permutation_invariance():
    q = RNG.standard_normal((4, 128))
    regs = _regions()
    a = attention.attend(q, regs, rotation.NONE, 0.5)
    b = attention.attend(q, regs[::-1], rotation.NONE, 0.5)
    d, K, V = regs[1]
    p = RNG.permutation(len(K))
    c = attention.attend(q, regs[:1] + [(d, K[p], V[p])] + regs[2:], rotation.NONE, 0.5)
    assert np.allclose(a, b, atol=1e-13) and np.allclose(a, c, atol=1e-13)


def test_brute_force_loops_tiny():
    # explicit per-element loops on a tiny case (N = 9, D = 8)
    q = RNG.standard_normal((1, 8))
    K, V = RNG.standard_normal((9, 8)), RNG.standard_normal((9, 8))
    s = [sum(q[0, c] * K[i, c] for c in range(8)) * 0.7 for i in range(9)]
    m = max(s)
    e = [np.exp(x - m) for x in s]
    tot = sum(e)
    o = [sum(e[i] / tot * V[i, c] for i in range(9)) for c in range(8)]
    assert np.allclose(attention.attend(q, [("exact", K[:4], V[:4]), ("exact", K[4:], V[4:])],
                                        rotation.NONE, 0.7)[0], o, atol=1e-14)
