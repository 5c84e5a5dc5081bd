"""Byte accounting of the oracle (test infrastructure).

KV cache math, "Bytes per token": kv_bytes_per_token = 2 x n_attn_layers x n_kv_heads x
head_dim x bytes_per_value; block formats by their block sizes (Q8_0 34 B / 32, Q4_0
18 B / 32, TBQ4 66 B / 128). SJ-KVaRN §2.1 (tq6_0: 98 B / 128), §3 (2,304 B of scales per
128-token record per KV head; effective-bits formula), §7.2 (allocation rule
body_bytes_per_token x (ctx - 4,224) + 259 MiB).
"""

from fractions import Fraction

# bytes per value, exact
BYTES_PER_VALUE = {
    "f16": Fraction(2),
    "bf16": Fraction(2),
    "q8_0": Fraction(34, 32),
    "q4_0": Fraction(18, 32),
    "tbq4": Fraction(66, 128),
    "tq6_0": Fraction(98, 128),
    "tq5_0": Fraction(82, 128),
    "turbo3": Fraction(50, 128),
    "q5_1": Fraction(24, 32),
    "q5_0": Fraction(22, 32),
    "q6_0": Fraction(26, 32),
    # the pages name q4_1 without its size: reading, two fp16 (d, m) + 16 B of nibbles per 32
    "q4_1": Fraction(20, 32),
}


def kvarn_bytes_per_value(bits):
    """KVarN-b: 4096*b code bytes + 1,152 scale bytes per 128 x 256 tile."""
    return Fraction(4096 * bits + 1152, 128 * 256)


def bytes_per_value(fmt):
    if fmt.startswith("kvarn"):
        return kvarn_bytes_per_value(int(fmt[5:]))
    return BYTES_PER_VALUE[fmt]


def kv_bytes_per_token(n_layers, n_kv_heads, head_dim, k_fmt, v_fmt=None):
    """Closed form: n_layers x n_kv_heads x head_dim x (bytes_K + bytes_V) per value."""
    v_fmt = k_fmt if v_fmt is None else v_fmt
    return n_layers * n_kv_heads * head_dim * (bytes_per_value(k_fmt) + bytes_per_value(v_fmt))


def record_bytes(fmt, head_dim):
    """Bytes of one 128-token body record of one KV head (K or V)."""
    return int(128 * head_dim * bytes_per_value(fmt))


def effective_bits(n_tokens, tail_tokens, body_bits):
    """SJ-KVaRN §3: [(N - 128 - t) body + t 6.125 + 128 (6.125 + 16)] / N."""
    N, t = Fraction(n_tokens), Fraction(tail_tokens)
    body = Fraction(body_bits)
    return ((N - 128 - t) * body + t * Fraction(49, 8) + 128 * (Fraction(49, 8) + 16)) / N


def allocation_rule_bytes(body_bytes_per_token, ctx):
    """SJ-KVaRN §7.2: body bytes/token x (ctx - 4,224) + 259 MiB."""
    return body_bytes_per_token * (ctx - 4224) + 259 * 1024 * 1024
