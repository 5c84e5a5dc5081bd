"""Pins of the oracle's byte accounting against numbers printed on the pages — CPU only."""

import json
import os
from fractions import Fraction

from oracle import sizes

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))
GB = 1024 ** 3
MIB = 1024 ** 2


def test_sj_f16_and_q8():
    g = G["sj_f16_bytes_per_token"]
    bpt = sizes.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"], "f16")
    assert bpt == g["value"]
    ctx = G["sj_f16_gb_at_110592"]["ctx"]
    assert round(float(bpt * ctx / GB), 2) == G["sj_f16_gb_at_110592"]["value"]
    assert round(float(sizes.kv_bytes_per_token(16, 4, 256, "q8_0") * ctx / GB), 2) == G["sj_q8_gb_at_110592"]["value"]


def test_sj_tail_ring_cost():
    g = G["sj_tail_mib_per_4096"]
    assert sizes.kv_bytes_per_token(16, 4, 256, "tq6_0") * 4096 == g["tq6_0"] * MIB
    assert sizes.kv_bytes_per_token(16, 4, 256, "f16") * 4096 == g["f16"] * MIB


def test_sj_scale_overhead():
    g = G["sj_scale_bits"]
    assert 2 * 1152 == g["bytes_per_record_per_head"]
    assert Fraction(g["bytes_per_record_per_head"] * 8, 2 * 128 * 256) == Fraction(g["bits_per_value"])
    assert sizes.record_bytes("kvarn4", 256) == 17536
    assert sizes.record_bytes("kvarn5", 512) == 2 * (20480 + 1152)


def _alloc_bits(kb, vb, ctx):
    body = 16 * 4 * (4096 * (kb + vb) + 2304) // 128            # bytes per token, 16 L x 4 H x 256
    total = sizes.allocation_rule_bytes(body, ctx)
    return total, total * 8 / (ctx * 16 * 2048)


def test_sj_allocation_rule_110592():
    g = G["sj_alloc_110592"]
    total, bits = _alloc_bits(4, 4, 110592)
    assert round(total / GB, 2) == g["4/4"]["gb"] and round(bits, 2) == g["4/4"]["bits"]
    assert round(_alloc_bits(3, 3, 110592)[1], 2) == g["3/3"]["bits"]
    assert round(_alloc_bits(3, 2, 110592)[1], 2) == g["3/2"]["bits"]


def test_sj_allocation_rule_204800():
    g = G["sj_alloc_204800"]
    total, bits = _alloc_bits(3, 2, 204800)
    assert round(total / GB, 2) == g["3/2"]["gb"] and round(bits, 2) == g["3/2"]["bits_rule"]
    assert round(_alloc_bits(4, 4, 204800)[1], 2) == g["4/4"]["bits"]
    assert round(_alloc_bits(3, 3, 204800)[1], 2) == g["3/3"]["bits"]


def test_sj_tq5_turbo4_average():
    b = (sizes.bytes_per_value("tq5_0") + sizes.bytes_per_value("tbq4")) * 8 / 2
    assert b == Fraction(37, 8)          # 4.625, printed 4.63 (rounded half up)
    assert abs(float(b) - G["sj_tq5_turbo4_bits"]["value"]) <= 0.005 + 1e-12


def test_hal_bytes_per_token():
    g = G["hal_f16_kib_per_token"]
    assert sizes.kv_bytes_per_token(48, 8, 128, "f16") == g["value"] * 1024
    c = G["hal_boot_cells"]
    assert c["cells"] * sizes.kv_bytes_per_token(48, 8, 128, "f16") == c["mib"] * MIB
    t = G["hal_kib_per_token"]
    for key, kib in t.items():
        if key == "cite":
            continue
        k, v = key.split("/")
        assert sizes.kv_bytes_per_token(48, 8, 128, k, v) == kib * 1024, key
    for ctx, row in G["hal_kv_mib"].items():
        if ctx == "cite":
            continue
        for key, mib in row.items():
            k, v = key.split("/")
            assert sizes.kv_bytes_per_token(48, 8, 128, k, v) * int(ctx) == mib * MIB


def test_math_tbq4_worked_example():
    g = G["math_tbq4"]
    bpt = g["mib"] * MIB // g["ctx"]
    assert bpt == g["bytes_per_token"]
    assert Fraction(bpt) / Fraction(66, 128) == g["values_per_token"]
    # 32,768 values per token = 2 x 16 layers x 4 heads x 256: the long-context config's shape
    assert sizes.kv_bytes_per_token(16, 4, 256, "tbq4") == g["bytes_per_token"]
    row = G["math_table_kib_per_token"]
    for fmt in ("f16", "q8_0", "q4_0", "tbq4", "turbo3"):
        assert Fraction(row[fmt]).limit_denominator(4) * 1024 == 32768 * sizes.bytes_per_value(fmt)
    gib = G["math_table_262k_gib"]
    for fmt in ("f16", "q8_0", "q4_0", "tbq4", "turbo3"):
        assert 32768 * sizes.bytes_per_value(fmt) * 262144 == Fraction(gib[fmt]).limit_denominator(8) * GB


def test_tail_page_persistent_kv():
    g = G["tail_persistent_mib_64k"]
    cells = g["bf16"] * MIB // 65536                  # 65,792 cells of 16 L x 2,048 values
    for fmt in ("q4_0", "q5_0", "q6_0", "q8_0"):
        assert float(cells * 16 * 2048 * sizes.bytes_per_value(fmt) / MIB) == g[fmt]


def test_effective_bits_formula_endpoints():
    # SJ-KVaRN section 3: with no body (N = 128 + t) only the tail and the sink count
    t = 4096
    assert sizes.effective_bits(128 + t, t, 4.28125) == (t * Fraction(49, 8) + 128 * (Fraction(49, 8) + 16)) / (128 + t)
    # at very long context the body rate dominates
    assert abs(float(sizes.effective_bits(10 ** 9, 4096, 4.28125)) - 4.28125) < 1e-4
