"""Decode attention of the oracle (test infrastructure), in fp64.

The plain definition over exactly the values the cache holds: positions in the exact
regions (sink, exact tail, exact journal) use the raw query and the stored K/V; positions
in the rotated regions (body, tq6_0 ring span) use the rotated query R q and the
dequantized rotated K/V, whose weighted sum is rotated back once (KV cache math,
"rotate first": q.k = (Hq).(Hk); the output is rotated back once at the end). All
positions share one softmax (KV Cache Precision Tail §2: "the two attention results are
combined under one softmax").

``region_partials`` + ``lse_merge`` restate the same result as per-region partial
softmaxes merged by log-sum-exp; tests check the two agree.
"""

import numpy as np

from .rotation import rotate_f64


def attend(q, regions, rot_kind, scale):
    """q [G, D]; regions: list of (domain, K [n, D], V [n, D]), domain 'exact' | 'rot'.

    Returns o [G, D] (fp64): softmax(scale * q_dom K^T) applied to V, rotated regions
    mapped back with R^T.
    """
    q = np.asarray(q, dtype=np.float64)
    q_rot = rotate_f64(q, rot_kind)
    scores, values, dom = [], [], []
    for domain, K, V in regions:
        K = np.asarray(K, dtype=np.float64)
        V = np.asarray(V, dtype=np.float64)
        if K.shape[0] == 0:
            continue
        qd = q if domain == "exact" else q_rot
        scores.append(scale * (qd @ K.T))
        values.append(V)
        dom.append(domain)
    s = np.concatenate(scores, axis=1)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    p = e / e.sum(axis=1, keepdims=True)
    o_exact = np.zeros_like(q)
    o_rot = np.zeros_like(q)
    col = 0
    for V, domain in zip(values, dom):
        n = V.shape[0]
        contrib = p[:, col:col + n] @ V
        if domain == "exact":
            o_exact += contrib
        else:
            o_rot += contrib
        col += n
    return o_exact + rotate_f64(o_rot, rot_kind, inverse=True)


def region_partials(q, regions, rot_kind, scale):
    """Per region: (domain, m [G], l [G], o_unnormalised [G, D]) with o = sum e^{s-m} v."""
    q = np.asarray(q, dtype=np.float64)
    q_rot = rotate_f64(q, rot_kind)
    out = []
    for domain, K, V in regions:
        K = np.asarray(K, dtype=np.float64)
        V = np.asarray(V, dtype=np.float64)
        if K.shape[0] == 0:
            continue
        qd = q if domain == "exact" else q_rot
        s = scale * (qd @ K.T)
        m = s.max(axis=1)
        e = np.exp(s - m[:, None])
        out.append((domain, m, e.sum(axis=1), e @ V))
    return out


def lse_merge(partials, rot_kind):
    """m* = max m_c; l* = sum e^{m_c - m*} l_c; o = (sum_exact w o_c + R^T sum_rot w o_c) / l*."""
    m_star = np.max(np.stack([p[1] for p in partials]), axis=0)
    l_star = np.zeros_like(m_star)
    o_exact = np.zeros_like(partials[0][3])
    o_rot = np.zeros_like(partials[0][3])
    for domain, m, l, o in partials:
        w = np.exp(m - m_star)
        l_star += w * l
        if domain == "exact":
            o_exact += w[:, None] * o
        else:
            o_rot += w[:, None] * o
    return (o_exact + rotate_f64(o_rot, rot_kind, inverse=True)) / l_star[:, None]
