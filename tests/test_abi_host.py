"""The C-ABI library on the host: it loads, exports every declared symbol, derives the same
format constants as the oracle on its own, and sizes configs like the oracle — CPU only
(no GPU call is made)."""

import os
import re

import numpy as np
import pytest

from oracle import sizes, tables
from quantized_kv_cache_gb300 import build, configs, _lib
from quantized_kv_cache_gb300.runner import prefill_plan

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _declared():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"^(?:kvq_status|const char\*)\s+(\w+)\s*\(", txt, re.M)
    return names


def test_every_declared_symbol_is_exported(lib):
    decl = _declared()
    assert len(decl) >= 15
    for name in decl:
        assert hasattr(lib, name), name
    assert set(decl) == set(_lib.exported_symbols())


def test_library_tables_equal_oracle_tables(lib):
    cent, bnd, words = _lib.kv_format_tables()
    oc, ob = tables.tbq4_tables()
    assert np.array_equal(np.array(cent, np.float32), oc)
    assert np.array_equal(np.array(bnd, np.float32), ob)
    assert tuple(words) == tables.sign_words()
    c3, b3 = _lib.kv_format_tables_turbo3()
    oc3, ob3 = tables.tbq3_tables()
    assert np.array_equal(np.array(c3, np.float32), oc3)
    assert np.array_equal(np.array(b3, np.float32), ob3)


@pytest.mark.parametrize("name", list(configs.WORKLOADS))
def test_bytes_per_token_matches_oracle(lib, name):
    w = configs.WORKLOADS[name]
    b = _lib.kv_bytes_per_token(w.config())
    body = sizes.kv_bytes_per_token(w.n_layers, w.n_kv_heads, w.head_dim, w.k_body, w.v_body)
    assert b["body_bytes_per_token"] == body
    assert b["f16_bytes_per_token"] == sizes.kv_bytes_per_token(w.n_layers, w.n_kv_heads, w.head_dim, "f16")
    jfmt = w.journal
    jb = sizes.kv_bytes_per_token(w.n_layers, w.n_kv_heads, w.head_dim, jfmt)
    assert b["journal_bytes_per_slot"] == jb
    pool, ws = _lib.kv_required_bytes(w.config())
    assert pool == b["pool_bytes"] and pool >= body * max(w.contexts) and ws > 0


def test_named_bytes_per_token_pins(lib):
    # KV cache math worked example: TBQ4 at 32,768 values/token = 16,896 B; HAL #582 §1: 78 KiB
    assert _lib.kv_bytes_per_token(configs.WORKLOADS["longctx_tbq4"].config())["body_bytes_per_token"] == 16896
    assert _lib.kv_bytes_per_token(configs.WORKLOADS["fa14b_q8q4"].config())["body_bytes_per_token"] == 78 * 1024
    assert _lib.kv_bytes_per_token(configs.WORKLOADS["hybrid27b_kvarn44"].config())["f16_bytes_per_token"] == 65536


def test_kvarn_widths_bytes_per_token(lib):
    """KVarN-b bodies of any width (and K / V widths that differ): the library's bytes per token
    are the oracle's closed form (SJ-KVaRN §3: 4,096 b code bytes + 1,152 B of scales per tile)."""
    from oracle import sizes
    base = configs.WORKLOADS["hybrid27b_kvarn44"]
    for kb, vb in ((2, 2), (3, 3), (3, 2), (6, 6), (8, 8), (8, 6), (4, 5)):
        c = base.config()
        c.k_body, c.v_body = _lib.FMT_NAMES[f"kvarn{kb}"], _lib.FMT_NAMES[f"kvarn{vb}"]
        got = _lib.kv_bytes_per_token(c)["body_bytes_per_token"]
        assert got == sizes.kv_bytes_per_token(16, 4, 256, f"kvarn{kb}", f"kvarn{vb}")
    c = base.config()
    c.k_body, c.v_body = _lib.KVARN3, _lib.KVARN2
    assert _lib.kv_bytes_per_token(c)["body_bytes_per_token"] == 11392     # the pages' 3/2 cache


@pytest.mark.parametrize("field,value", [("head_dim", 192), ("n_q_heads", 4 * 32), ("ring_capacity", 1000),
                                         ("tail_fmt", _lib.TQ6_0), ("k_body", _lib.F16), ("v_body", _lib.TBQ4),
                                         ("kvarn_balance", 2), ("kvarn_balance", -1)])
def test_invalid_configs_refused(lib, field, value):
    c = configs.WORKLOADS["hybrid27b_kvarn44"].config()
    setattr(c, field, value)
    with pytest.raises(_lib.KVQError) as e:
        _lib.kv_required_bytes(c)
    assert e.value.code == 1


def test_kvarn_balance_rules_accepted(lib):
    # both balancing rules take the same pool: the records have one layout
    c = configs.WORKLOADS["hybrid27b_kvarn44"].config()
    sizes = []
    for rule in (_lib.KVARN_BALANCE["final16"], _lib.KVARN_BALANCE["best8"]):
        c.kvarn_balance = rule
        sizes.append(_lib.kv_required_bytes(c))
    assert sizes[0] == sizes[1]


def test_kvarn_needs_256_multiple(lib):
    c = configs.WORKLOADS["hybrid27b_kvarn44"].config()
    c.head_dim = 128
    with pytest.raises(_lib.KVQError):
        _lib.kv_required_bytes(c)


def _simulate(w, n0):
    n, S = 0, 128
    for c, seal in prefill_plan(w, n0):
        n += c
        assert configs.journal_len(n, S) <= w.ring
        if seal:
            S += 128 * configs.groups_to_seal(n, S, w.keep)
    return n, S


def test_prefill_plans_reach_stated_states():
    w = configs.WORKLOADS["hybrid27b_kvarn44"]
    assert _simulate(w, 32768) == (32768, 24704)          # 192 groups sealed, journal 8,064
    w = configs.WORKLOADS["fa14b_q8q4"]
    assert _simulate(w, 131072) == (131072, 130048)       # 1,015 groups, journal 1,024
    w = configs.WORKLOADS["widehead_kvarn55"]
    for n0 in w.contexts:
        assert 8192 <= n0 <= 16384
        assert _simulate(w, n0) == (n0, 128 + 128 * ((n0 - 2176) // 128))
    w = configs.WORKLOADS["longctx_tbq4"]
    for n0 in w.contexts:
        assert _simulate(w, n0) == (n0, n0 - 20480)       # 128 groups + 4,096 unsealed
    w = configs.WORKLOADS["tiny_tbq4"]
    assert _simulate(w, 1023) == (1023, 128)


def test_decode_seal_points():
    # hybrid: journal 8,064 + 128 steps reaches 8,192 -> seal 32 groups (SJ-KVaRN §4.3)
    w = configs.WORKLOADS["hybrid27b_kvarn44"]
    n, S = 32768, 24704
    for step in range(256):
        n += 1
        if configs.should_seal(w, n, S):
            assert step == 127 and configs.groups_to_seal(n, S, w.keep) == 32
            S += 128 * 32
    # longctx bulk seal after step 16: 128 groups per sequence
    w = configs.WORKLOADS["longctx_tbq4"]
    for n0 in w.contexts:
        assert configs.groups_to_seal(n0 + 16, n0 - 20480, w.keep) == 128


def test_bench_streaming_table_matches_the_dispatch_table():
    """bench.py counts launches by the streaming decode kernel's instances; they must be the
    instances kernels_body.cu dispatches to (KVQ_BODY_CASE lines)."""
    import re
    import bench
    src = open(os.path.join(os.path.dirname(__file__), "..", "quantized_kv_cache_gb300", "csrc",
                            "kernels_body.cu")).read()
    names = {"KVQ_TBQ4": "tbq4", "KVQ_Q8_0": "q8_0", "KVQ_Q4_0": "q4_0", "KVQ_KVARN2": "kvarn2",
             "KVQ_KVARN3": "kvarn3", "KVQ_KVARN4": "kvarn4", "KVQ_KVARN5": "kvarn5", "KVQ_Q5_1": "q5_1",
             "KVQ_TQ5_0": "tq5_0"}
    cases = set()
    # (D, NQ, K reader, V reader, K bits, V bits, K format, V format, region kinds)
    for m in re.finditer(r"KVQ_BODY_CASE\((\d+), (\d+), \w+, \w+, \d, \d, (\w+), (\w+), \d+\)", src):
        cases.add((int(m.group(1)), int(m.group(2)), names[m.group(3)], names[m.group(4)]))
    assert cases and cases == bench.STREAMING
