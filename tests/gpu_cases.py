"""Shared builders of the GPU parity tests: one small cache per format family, driven
identically through the C ABI (GPU) and through the oracle's region model (CPU).

Shapes span several decode tiles and chunks, ragged region ends, ring wrap-around and
several layers / sequences, yet the oracle finishes each family in seconds.
"""

from dataclasses import dataclass
from typing import List

import numpy as np

from oracle.cache import HeadCache, HeadConfig
from quantized_kv_cache_gb300 import synth, _lib


@dataclass
class Family:
    name: str
    D: int
    H: int
    Hq: int
    k_body: str
    v_body: str
    journal: str
    tail_fmt: str
    T: int
    R: int
    contexts: List[int]
    keep: int
    steps: int
    L: int = 2
    seed: int = 9
    n_out: int = 4
    factor: float = 16.0
    balance: str = "final16"      # KVarN balancing: "final16" or "best8"

    def config(self):
        c = _lib.kvq_config()
        c.n_layers, c.n_kv_heads, c.head_dim, c.n_q_heads = self.L, self.H, self.D, self.Hq
        c.max_seqs = len(self.contexts) + 1
        c.max_ctx = max(self.contexts) + self.steps + 256
        c.k_body, c.v_body = _lib.FMT_NAMES[self.k_body], _lib.FMT_NAMES[self.v_body]
        c.journal, c.tail_fmt = _lib.FMT_NAMES[self.journal], _lib.FMT_NAMES[self.tail_fmt]
        c.tail, c.ring_capacity, c.softmax_scale = self.T, self.R, 0.0
        c.kvarn_balance = _lib.KVARN_BALANCE[self.balance]
        return c

    def head_config(self):
        return HeadConfig(self.D, self.k_body, self.v_body, self.journal, self.tail_fmt, self.T, self.R,
                          self.balance)


FAMILIES = {
    "tbq4_f16": Family("tbq4_f16", 128, 2, 4, "tbq4", "tbq4", "f16", "f16", T=128, R=1024,
                       contexts=[900, 1413], keep=128, steps=3),
    "kvarn4_ring": Family("kvarn4_ring", 256, 2, 12, "kvarn4", "kvarn4", "tq6_0", "f16", T=64, R=1024,
                          contexts=[700, 1555], keep=256, steps=3, factor=16.0, n_out=8),
    "q8q4_bf16": Family("q8q4_bf16", 128, 2, 10, "q8_0", "q4_0", "bf16", "bf16", T=256, R=768,
                        contexts=[1000, 1790], keep=256, steps=3, factor=20.0),
    "kvarn5_wide": Family("kvarn5_wide", 512, 1, 16, "kvarn5", "kvarn5", "f16", "f16", T=256, R=768,
                          contexts=[777, 1200], keep=256, steps=2, factor=12.0, n_out=16),
    "tbq4_ring": Family("tbq4_ring", 256, 2, 12, "tbq4", "tbq4", "tq6_0", "f16", T=96, R=896,
                        contexts=[640, 1900], keep=384, steps=3, n_out=8),
    # KVarN widths without a streaming instance (the generic decode path): 3-bit keys with
    # 2-bit values on a tq6_0 ring, and 8-bit keys with 6-bit values on an F16 journal
    "kvarn32_ring": Family("kvarn32_ring", 256, 2, 8, "kvarn3", "kvarn2", "tq6_0", "f16", T=64, R=768,
                           contexts=[650, 1300], keep=256, steps=2, factor=16.0, n_out=8),
    "kvarn86_f16": Family("kvarn86_f16", 256, 1, 6, "kvarn8", "kvarn6", "f16", "f16", T=128, R=768,
                          contexts=[900, 1250], keep=128, steps=2, factor=16.0, n_out=8),
    # the other 32-value block formats (generic decode path): the tier ladder's floor rung
    # q5_1 K / q4_0 V on a BF16 journal, q6_0 K / q4_1 V and q5_0 K / q5_0 V on F16 journals
    "q51q40_bf16": Family("q51q40_bf16", 128, 2, 10, "q5_1", "q4_0", "bf16", "bf16", T=256, R=768,
                          contexts=[900, 1333], keep=256, steps=2, factor=20.0),
    "q60q41_f16": Family("q60q41_f16", 128, 1, 4, "q6_0", "q4_1", "f16", "f16", T=128, R=768,
                         contexts=[800, 1201], keep=128, steps=2, factor=12.0),
    "q50q50_f16": Family("q50q50_f16", 256, 1, 2, "q5_0", "q5_0", "f16", "f16", T=64, R=512,
                         contexts=[700], keep=64, steps=2, factor=16.0, n_out=8),
    # the rotated comparators (generic decode path): tq5_0 K with TBQ4 (turbo4) V on a tq6_0
    # ring, and turbo3 K and V on an F16 journal
    "tq50tbq4_ring": Family("tq50tbq4_ring", 256, 2, 8, "tq5_0", "tbq4", "tq6_0", "f16", T=96, R=896,
                            contexts=[700, 1300], keep=384, steps=2, n_out=8),
    "turbo3_f16": Family("turbo3_f16", 128, 2, 4, "turbo3", "turbo3", "f16", "f16", T=128, R=1024,
                         contexts=[900, 1413], keep=128, steps=2),
    # the KVarN reference configuration's balancing (8 passes, the best state kept): 4/4 on a
    # tq6_0 ring (streaming decode instance) and 3/2 on an F16 journal
    "kvarn4b8_ring": Family("kvarn4b8_ring", 256, 2, 12, "kvarn4", "kvarn4", "tq6_0", "f16", T=64, R=1024,
                            contexts=[720, 1500], keep=256, steps=2, n_out=8, seed=13, balance="best8"),
    "kvarn32b8_f16": Family("kvarn32b8_f16", 256, 1, 8, "kvarn3", "kvarn2", "f16", "f16", T=128, R=768,
                            contexts=[850, 1290], keep=128, steps=2, n_out=8, seed=14, balance="best8"),
}


def inputs(f: Family, layer, seq, pos0, n):
    k = synth.kv_block(f.seed, synth.T_K, layer, seq, pos0, n, f.H, f.D, f.n_out, f.factor)
    v = synth.kv_block(f.seed, synth.T_V, layer, seq, pos0, n, f.H, f.D)
    return k, v


def prefill_chunks(f: Family, n0):
    """Append chunks of at most 300 positions, sealing (keep) after each so the journal
    never exceeds R; leaves the seal state the policy 'seal whenever possible' gives."""
    out, n, S = [], 0, 128
    while n < n0:
        c = min(300, n0 - n, f.R - (max(n, 128) - S))
        n += c
        lim = n - f.keep - S
        g = lim // 128 if lim >= 128 else 0
        S += 128 * g
        out.append(c)
    return out


class Pair:
    """The GPU cache and the per-(layer, seq, head) oracle caches of one family."""

    def __init__(self, f: Family, device=0):
        import torch
        from quantized_kv_cache_gb300 import KVCache
        self.f, self.torch = f, torch
        self.gpu = KVCache(f.config(), device)
        self.seqs = list(range(len(f.contexts)))
        self.hc = {(l, s, h): HeadCache(f.head_config()) for l in range(f.L) for s in self.seqs for h in range(f.H)}
        self.dev = torch.device("cuda", device)

    def append(self, layer, seqs, pos0s, n):
        ks, vs = [], []
        for s, p0 in zip(seqs, pos0s):
            k, v = inputs(self.f, layer, s, p0, n)
            ks.append(k)
            vs.append(v)
            for h in range(self.f.H):
                self.hc[(layer, s, h)].append(k[:, h], v[:, h])
        K = self.torch.from_numpy(np.stack(ks)).to(self.dev)
        V = self.torch.from_numpy(np.stack(vs)).to(self.dev)
        self.gpu.append(layer, seqs, K, V)

    def seal(self, layer, seqs, keep):
        g = self.gpu.seal(layer, seqs, keep)
        go = 0
        for s in seqs:
            for h in range(self.f.H):
                n = self.hc[(layer, s, h)].seal(keep)
            go += n
        return g, go

    def prefill(self):
        for layer in range(self.f.L):
            for s, n0 in zip(self.seqs, self.f.contexts):
                pos = 0
                for c in prefill_chunks(self.f, n0):
                    self.append(layer, [s], [pos], c)
                    pos += c
                    self.seal(layer, [s], self.f.keep)

    def region_bytes(self, layer, seq, head, which, region):
        """Bytes of one region's storage, sliced out of the pool tensor that holds it."""
        ptr, nb = _lib.kv_region_ptr(self.gpu.h, layer, seq, head, which, region)
        off = ptr - self.gpu.pool.data_ptr()
        assert 0 <= off and off + nb <= self.gpu.pool_bytes
        self.torch.cuda.synchronize()
        return self.gpu.pool[off:off + nb].cpu().numpy()

    def dequant(self, layer, seq, head, which, p0, n):
        out = self.torch.empty((n, self.f.D), dtype=self.torch.float32, device=self.dev)
        _lib.kv_dequant(self.gpu.h, layer, seq, head, which, p0, n, out.data_ptr())
        self.torch.cuda.synchronize()
        return out.cpu().numpy()

    def attend(self, layer, seqs, q_np):
        q = self.torch.from_numpy(q_np).to(self.dev)
        out = self.torch.empty_like(q)
        self.gpu.decode_attn(layer, seqs, q, out)
        self.torch.cuda.synchronize()
        return out.cpu().numpy()
