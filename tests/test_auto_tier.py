"""The auto KV-tier policy (HAL #582 §5 P1) through the C ABI, on the host.

Pins: the page's validated example (Qwen2.5-14B-1M: 48 layers, 8 KV heads x 128, a
32,768-position cache) prints the whole-cache costs 3,264 MiB for q8_0/q8_0 and 2,496 MiB for
q8_0/q4_0, the budgets 3,328 / 2,728 / 2,128 MiB that the vram targets 20,000 / 19,400 /
18,800 MiB leave, and the rung each budget takes (q8_0/q8_0, q8_0/q4_0, then the floor rung
q5_1/q4_0 at 2,016 MiB). The f16 cost is the page's 192 KiB per token. Costs also equal the
oracle's closed-form bytes per token.
"""

import pytest

from oracle import sizes
from quantized_kv_cache_gb300 import _lib

MiB = 1 << 20


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def shape(L=48, H=8, D=128):
    c = _lib.kvq_config()
    c.n_layers, c.n_kv_heads, c.head_dim = L, H, D
    return c


def test_page_example_costs_and_choices(lib):
    c = shape()
    k, v, cost, fits = _lib.kv_auto_tier(c, 32768, 3328 * MiB)
    assert (k, v, fits) == (_lib.Q8_0, _lib.Q8_0, True) and cost == 3264 * MiB
    k, v, cost, fits = _lib.kv_auto_tier(c, 32768, 2728 * MiB)
    assert (k, v, fits) == (_lib.Q8_0, _lib.Q4_0, True) and cost == 2496 * MiB
    # the page's last rung: 18,800 MiB target -> q5_1/q4_0, 2,016 MiB fits 2,128
    k, v, cost, fits = _lib.kv_auto_tier(c, 32768, 2128 * MiB)
    assert (k, v, fits) == (_lib.Q5_1, _lib.Q4_0, True) and cost == 2016 * MiB
    k, v, cost, fits = _lib.kv_auto_tier(c, 32768, 2000 * MiB)     # the floor does not fit either
    assert (k, v, fits) == (_lib.Q5_1, _lib.Q4_0, False) and cost == 2016 * MiB
    k, v, cost, fits = _lib.kv_auto_tier(c, 32768, 6144 * MiB)
    assert (k, v, fits) == (_lib.F16, _lib.F16, True) and cost == 32768 * 192 * 1024


def test_budget_rule_reproduces_the_page_budgets(lib):
    # one resident figure explains all three of the page's (target, budget) pairs
    resident = (20000 - 3328) * MiB - 1536 * MiB
    for target, budget in ((20000, 3328), (19400, 2728), (18800, 2128)):
        assert _lib.kv_tier_budget(96 * 1024 * MiB, resident, target * MiB) == budget * MiB
    # no target: the free bytes cap it; nothing left: 0
    assert _lib.kv_tier_budget(8000 * MiB, 1000 * MiB) == (8000 - 1000 - 1536) * MiB
    assert _lib.kv_tier_budget(1000 * MiB, 1000 * MiB) == 0


@pytest.mark.parametrize("L,H,D,tokens", [(48, 8, 128, 32768), (16, 4, 256, 262144), (10, 2, 512, 12345),
                                          (1, 1, 128, 1), (60, 8, 128, 0)])
def test_costs_equal_oracle_bytes_per_token(lib, L, H, D, tokens):
    c = shape(L, H, D)
    for budget, pair in ((1 << 62, ("f16", "f16")), (0, ("q5_1", "q4_0"))):
        k, v, cost, fits = _lib.kv_auto_tier(c, tokens, budget)
        assert cost == tokens * sizes.kv_bytes_per_token(L, H, D, *pair)
        assert fits == (cost <= budget)


def test_ladder_order_and_refusals(lib):
    c = shape()
    per_token = [sizes.kv_bytes_per_token(48, 8, 128, *p) for p in (("f16", "f16"), ("q8_0", "q8_0"),
                                                                    ("q8_0", "q4_0"), ("q5_1", "q4_0"))]
    assert per_token == sorted(per_token, reverse=True)           # least compression first
    for budget in range(0, 7000 * MiB, 97 * MiB):
        k, v, cost, fits = _lib.kv_auto_tier(c, 32768, budget)
        # the first rung that fits, or the floor
        want = next((i for i, b in enumerate(per_token) if 32768 * b <= budget), 3)
        assert cost == 32768 * per_token[want]
    bad = shape(0)
    with pytest.raises(_lib.KVQError):
        _lib.kv_auto_tier(bad, 10, 10)
    with pytest.raises(_lib.KVQError):
        _lib.kv_auto_tier(c, -1, 10)
