"""The five workloads this package is measured and checked on, by name and shape.

Each entry gives the cache configuration (``kvq_config``) and the run recipe: how the
initial cache state is built (positions, sealed end), how many decode steps run, the seal
policy (``keep`` and the journal length that triggers a seal) and the synthetic input
recipe (seed, K outlier channels and factor).

- tiny_tbq4: 1 sequence, 1 layer, 2 KV heads x 128, 4 query heads; TBQ4 body, F16
  journal with a 128-position tail; 1,023 positions appended, then one step appends
  position 1,023, seals 6 groups and attends over 1,024 = 128 sink + 768 body + 128 tail.
- hybrid27b_kvarn44: 16 layers, 4 KV heads x 256, 24 query heads, 1 sequence at 32,768
  positions; KVarN 4/4 body, tq6_0 ring of 8,448 positions, 1,024-position F16 exact tail;
  seal every group older than the newest 4,096 when the journal reaches 8,192 (SJ-KVaRN
  §4.3); 256 decode steps.
- fa14b_q8q4: 48 layers, 8 KV heads x 128, 40 query heads, 1 sequence at 131,072; Q8_0 K,
  Q4_0 V, BF16 journal that is the 1,024-position exact tail (ring of 5,248 positions so
  prefill can append 4,096 at a time); 64 decode steps.
- widehead_kvarn55: 8 sequences with seeded contexts in [8,192, 16,384], 10 full-attention
  layers, 2 KV heads x 512 (two 256-point halves), 32 query heads; KVarN 5/5, F16 journal /
  2,048-position tail; 128 decode steps.
- longctx_tbq4: 4 sequences at 262,144 / 196,608 / 131,072 / 65,536, 16 layers, 4 KV
  heads x 256, 24 query heads; TBQ4 body (16,896 B per position), tq6_0 ring, 1,024-position
  tail; each sequence starts with 128 groups + 4,096 positions unsealed; 32 decode steps
  with a bulk seal of 4 x 128 = 512 groups per layer after step 16.

A sixth workload measures the KVarN widths beyond 4 and 5 (SJ-KVaRN §7, the 3/2 cache of the
12 GB-card run, here with the scalar body, whose records take as many bytes as the trellis ones):
- hybrid27b_kvarn32_200k: the hybrid27b shape at 204,800 positions with KVarN 3-bit K and
  2-bit V, tq6_0 ring, the same seal policy; 64 decode steps.
And a seventh the block formats beyond Q8_0 / Q4_0 (the auto tier's floor rung, HAL #582 §5):
- fa14b_q51q40: the fa14b_q8q4 shape and policy with q5_1 K and q4_0 V.
An eighth the rotated comparator the pages measure SJ-KVaRN against (SJ-KVaRN §4.1):
- hybrid27b_tq50tbq4_110k: the hybrid27b shape and policy at 110,592 positions with tq5_0 K and
  TBQ4 (turbo4) V.
"""

from dataclasses import dataclass, field
from typing import List

from . import _lib
from . import synth


@dataclass
class Workload:
    name: str
    n_layers: int
    n_kv_heads: int
    head_dim: int
    n_q_heads: int
    k_body: str
    v_body: str
    journal: str
    tail_fmt: str
    tail: int
    ring: int
    contexts: List[int]
    steps: int
    seed: int
    n_out: int
    out_factor: float
    keep: int
    seal_trigger: int            # journal length that triggers a seal (0: seal whenever possible)
    prefill_unsealed: int = 0    # positions left unsealed after prefill (0: follow the seal policy)
    bulk_seal_step: int = -1     # decode step after which a bulk seal runs (-1: none)
    extra_ctx: int = 512

    @property
    def G(self):
        return self.n_q_heads // self.n_kv_heads

    def config(self, max_seqs=None, n_layers=None):
        c = _lib.kvq_config()
        c.n_layers = n_layers or self.n_layers
        c.n_kv_heads = self.n_kv_heads
        c.head_dim = self.head_dim
        c.n_q_heads = self.n_q_heads
        c.max_seqs = max_seqs or len(self.contexts)
        c.max_ctx = max(self.contexts) + self.steps + self.extra_ctx
        c.k_body = _lib.FMT_NAMES[self.k_body]
        c.v_body = _lib.FMT_NAMES[self.v_body]
        c.journal = _lib.FMT_NAMES[self.journal]
        c.tail_fmt = _lib.FMT_NAMES[self.tail_fmt]
        c.tail = self.tail
        c.ring_capacity = self.ring
        c.softmax_scale = 0.0
        return c


WORKLOADS = {
    "tiny_tbq4": Workload("tiny_tbq4", 1, 2, 128, 4, "tbq4", "tbq4", "f16", "f16", tail=128, ring=1024,
                          contexts=[1023], steps=1, seed=0, n_out=4, out_factor=16.0, keep=128,
                          seal_trigger=-1),
    "hybrid27b_kvarn44": Workload("hybrid27b_kvarn44", 16, 4, 256, 24, "kvarn4", "kvarn4", "tq6_0", "f16",
                                  tail=1024, ring=8448, contexts=[32768], steps=256, seed=1, n_out=8,
                                  out_factor=16.0, keep=4096, seal_trigger=8192),
    "fa14b_q8q4": Workload("fa14b_q8q4", 48, 8, 128, 40, "q8_0", "q4_0", "bf16", "bf16", tail=1024, ring=5248,
                           contexts=[131072], steps=64, seed=2, n_out=4, out_factor=20.0, keep=1024,
                           seal_trigger=0),
    "widehead_kvarn55": Workload("widehead_kvarn55", 10, 2, 512, 32, "kvarn5", "kvarn5", "f16", "f16", tail=2048,
                                 ring=6272, contexts=synth.context_lengths(3, 8, 8192, 16384), steps=128,
                                 seed=3, n_out=16, out_factor=12.0, keep=2048, seal_trigger=0),
    "longctx_tbq4": Workload("longctx_tbq4", 16, 4, 256, 24, "tbq4", "tbq4", "tq6_0", "f16", tail=1024,
                             ring=20608, contexts=[262144, 196608, 131072, 65536], steps=32, seed=4, n_out=8,
                             out_factor=16.0, keep=4096, seal_trigger=-2, prefill_unsealed=128 * 128 + 4096,
                             bulk_seal_step=16),
    "fa14b_q51q40": Workload("fa14b_q51q40", 48, 8, 128, 40, "q5_1", "q4_0", "bf16", "bf16", tail=1024, ring=5248,
                             contexts=[131072], steps=64, seed=6, n_out=4, out_factor=20.0, keep=1024,
                             seal_trigger=0),
    "hybrid27b_tq50tbq4_110k": Workload("hybrid27b_tq50tbq4_110k", 16, 4, 256, 24, "tq5_0", "tbq4", "tq6_0",
                                        "f16", tail=1024, ring=8448, contexts=[110592], steps=64, seed=7, n_out=8,
                                        out_factor=16.0, keep=4096, seal_trigger=8192),
    "hybrid27b_kvarn32_200k": Workload("hybrid27b_kvarn32_200k", 16, 4, 256, 24, "kvarn3", "kvarn2", "tq6_0",
                                       "f16", tail=1024, ring=8448, contexts=[204800], steps=64, seed=5, n_out=8,
                                       out_factor=16.0, keep=4096, seal_trigger=8192),
}


def record_bytes(fmt, head_dim):
    """Bytes of one 128-position body record of one KV head (K or V) in the given format."""
    return {"tbq4": 66 * head_dim, "q8_0": 136 * head_dim, "q4_0": 72 * head_dim, "q5_0": 88 * head_dim,
            "q6_0": 104 * head_dim, "q4_1": 80 * head_dim, "q5_1": 96 * head_dim, "turbo3": 50 * head_dim,
            "tq5_0": 82 * head_dim,
            **{f"kvarn{b}": (head_dim // 256) * (4096 * b + 1152) for b in (2, 3, 4, 5, 6, 8)}}[fmt]


def journal_len(n_tok, sealed):
    return max(n_tok, 128) - sealed


def groups_to_seal(n_tok, sealed, keep):
    lim = n_tok - keep - sealed
    return lim // 128 if lim >= 128 else 0


def should_seal(w: Workload, n_tok, sealed):
    """Seal policy after an append: returns True when kv_seal(keep=w.keep) should run.

    seal_trigger > 0: seal when the journal holds that many positions (adaptive tail,
    SJ-KVaRN §4.3); 0: seal whenever a full group older than ``keep`` exists; negative:
    never during decode (tiny_tbq4 seals once explicitly; longctx_tbq4 runs a bulk seal).
    """
    if w.seal_trigger > 0:
        return journal_len(n_tok, sealed) >= w.seal_trigger
    if w.seal_trigger == 0:
        return groups_to_seal(n_tok, sealed, w.keep) > 0
    return False
