"""Pins of the oracle's region model (append, seal, regions) — CPU only.

SJ-KVaRN §2.1 (sink, tq6_0 staging, exact tail, batched seal of full 128-token groups
older than the newest 4,096) and §4.3 (adaptive tail, one batch per ~4,096 tokens);
KV Cache Precision Tail §2 (exact recent region + quantized body under one softmax).
"""

import numpy as np
import pytest

from oracle import attention, rotation
from oracle.cache import HeadCache, HeadConfig, SINK
from quantized_kv_cache_gb300 import synth


def _fill(hc, n, seed=0, head=0, n_out=4, factor=16.0):
    D = hc.cfg.head_dim
    k = synth.kv_values(seed, synth.T_K, 0, 0, head, 0, n, D, n_out, factor)
    v = synth.kv_values(seed, synth.T_V, 0, 0, head, 0, n, D)
    hc.append(k, v)
    return k, v


def _positions(hc):
    return sum(len(K) for _, K, _ in hc.regions())


CFGS = {
    "tiny_tbq4": HeadConfig(128, "tbq4", "tbq4", "f16", "f16", tail=128, ring=512),
    "kvarn_ring": HeadConfig(256, "kvarn4", "kvarn4", "tq6_0", "f16", tail=64, ring=768),
    "q8q4_bf16": HeadConfig(128, "q8_0", "q4_0", "bf16", "bf16", tail=128, ring=512),
    "tbq4_ring": HeadConfig(256, "tbq4", "tbq4", "tq6_0", "f16", tail=32, ring=512),
    "kvarn5_wide": HeadConfig(512, "kvarn5", "kvarn5", "f16", "f16", tail=128, ring=512),
}


@pytest.mark.parametrize("name", list(CFGS))
def test_regions_partition_positions(name):
    hc = HeadCache(CFGS[name])
    _fill(hc, 50)
    assert _positions(hc) == 50 and hc.S == SINK
    _fill(hc, 600 - 50)
    assert _positions(hc) == 600
    g = hc.seal(keep=hc.cfg.tail)
    # groups sealed: every full group with S + 128 <= N - keep
    assert g == (600 - hc.cfg.tail - SINK) // 128
    assert hc.S == SINK + 128 * g and _positions(hc) == 600
    assert hc.seal(keep=hc.cfg.tail) == 0


def test_exact_regions_are_verbatim():
    hc = HeadCache(CFGS["kvarn_ring"])
    k, v = _fill(hc, 500)
    regs = hc.regions()
    assert np.array_equal(regs[0][1], k[:128].astype(np.float32))
    dom, Kt, Vt = regs[-1]
    assert dom == "exact" and np.array_equal(Kt, k[500 - 64:].astype(np.float32))
    assert np.array_equal(Vt, v[500 - 64:].astype(np.float32))


def test_bf16_journal_rounds_to_bf16():
    hc = HeadCache(CFGS["q8q4_bf16"])
    k, v = _fill(hc, 300)
    Kj = hc.regions()[-1][1]
    kf = k[128:].astype(np.float32)
    # bf16 keeps 8 significant bits: relative error <= 2^-8 (half an ulp), values bf16-representable
    assert np.all(np.abs(Kj - kf) <= np.abs(kf) * 2.0 ** -8)
    assert np.all((Kj.view(np.uint32) & 0xFFFF) == 0)


def test_journal_overflow_refused():
    hc = HeadCache(CFGS["tiny_tbq4"])
    _fill(hc, 128 + 512)
    with pytest.raises(OverflowError):
        hc.append(np.zeros((1, 128), np.float16), np.zeros((1, 128), np.float16))
    hc.seal(keep=128)
    hc.append(np.zeros((1, 128), np.float16), np.zeros((1, 128), np.float16))


def test_ring_wraparound_keeps_positions():
    cfg = CFGS["tbq4_ring"]
    hc = HeadCache(cfg)
    k, v = _fill(hc, 128 + 500)
    hc.seal(keep=32)            # seals 3 groups
    k2 = synth.kv_values(0, synth.T_K, 0, 0, 0, 628, 300, 256, 4, 16.0)
    v2 = synth.kv_values(0, synth.T_V, 0, 0, 0, 628, 300, 256)
    hc.append(k2, v2)           # wraps the 512-slot ring
    kk = np.concatenate([k, k2])
    # ring rows decode to the rotated inputs within tq6_0 error
    rows = hc.journal_rows("K", 700, 100)
    ref = rotation.rotate(kk[700:800].astype(np.float32), rotation.TBQ128)
    assert np.max(np.abs(rows - ref)) <= np.max(np.abs(ref)) / 31
    assert _positions(hc) == 928


@pytest.mark.parametrize("name", ["tiny_tbq4", "kvarn_ring", "q8q4_bf16", "kvarn5_wide"])
def test_cache_attention_close_to_unquantized(name):
    # Sanity of the whole model: attention over the cache regions is close to fp64 attention
    # over the raw fp16 inputs (quantization error only), with a sharp softmax.
    cfg = CFGS[name]
    hc = HeadCache(cfg)
    k, v = _fill(hc, 600, n_out=0)
    hc.seal(keep=cfg.tail)
    D = cfg.head_dim
    q = synth.q_values(0, 0, 0, 0, 4, D, q_scale=4.0 / np.sqrt(D)).astype(np.float64)
    scale = 1 / np.sqrt(D)
    o = attention.attend(q, hc.regions(), cfg.rot, scale)
    ref = attention.attend(q, [("exact", k.astype(np.float64), v.astype(np.float64))], rotation.NONE, scale)
    assert np.max(np.abs(o - ref)) < 0.05
