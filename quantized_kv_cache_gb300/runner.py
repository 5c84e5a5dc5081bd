"""Drives a workload through the C ABI: synthetic inputs in HBM, prefill, decode steps.

Host-side orchestration only (which call to make when, per the workload's seal policy);
every step of the method runs inside libkvq.so. Used by the benchmark, the GPU tests and
the smoke check.
"""

import numpy as np

from . import KVCache, synth
from ._lib import kvq_synth_fill
from .configs import Workload, journal_len, groups_to_seal, should_seal


class DeviceSynth:
    """Fills CUDA tensors with the same values ``synth`` draws on the host."""

    def __init__(self, w: Workload, device=0):
        import torch
        self.torch = torch
        self.w = w
        self.dev = torch.device("cuda", device)
        tab = synth.normal_table().view(np.int16)
        self.table = torch.from_numpy(tab.copy()).to(self.dev)
        H, D = w.n_kv_heads, w.head_dim
        self.k_factor = {}
        self.q_factor = torch.full((w.n_q_heads, D), float(np.float32(1.0 / np.sqrt(D))), dtype=torch.float32,
                                   device=self.dev)
        self._H, self._D = H, D

    def _kfactor(self, layer):
        if layer not in self.k_factor:
            w = self.w
            f = np.ones((self._H, self._D), np.float32)
            if w.n_out:
                for h in range(self._H):
                    f[h, synth.outlier_channels(w.seed, layer, h, self._D, w.n_out)] = np.float32(w.out_factor)
            self.k_factor[layer] = self.torch.from_numpy(f).to(self.dev)
        return self.k_factor[layer]

    def kv(self, tensor, layer, seq, pos0, n_pos, out, stream=0):
        """out: fp16 CUDA tensor with n_pos * H * D elements ([n_pos, H, D])."""
        keys = [synth.stream_key(self.w.seed, tensor, layer, seq, h) for h in range(self._H)]
        fac = self._kfactor(layer).data_ptr() if (tensor == synth.T_K and self.w.n_out) else 0
        kvq_synth_fill(out.data_ptr(), n_pos, self._H, self._D, keys, pos0, fac, self.table.data_ptr(), stream)

    def q(self, layer, seq, step, out, stream=0):
        """out: fp16 CUDA tensor [Hq, D] — the query of decode step ``step``."""
        keys = [synth.stream_key(self.w.seed, synth.T_Q, layer, seq, h) for h in range(self.w.n_q_heads)]
        kvq_synth_fill(out.data_ptr(), 1, self.w.n_q_heads, self._D, keys, step, self.q_factor.data_ptr(),
                       self.table.data_ptr(), stream)


def prefill_plan(w: Workload, n0, chunk_max=4096):
    """Chunks (n_tok, seal_after) that build the workload's starting state for a sequence
    with n0 positions: the decode seal policy applied during prefill, or for longctx the
    state 'all but the newest prefill_unsealed positions sealed'."""
    plan, n, S = [], 0, 128
    if w.prefill_unsealed:
        phase1 = n0 - (w.prefill_unsealed - w.keep)
        while n < n0:
            c = min(chunk_max, n0 - n) if n >= phase1 else min(chunk_max, phase1 - n)
            n += c
            seal = n <= phase1
            if seal:
                S += 128 * groups_to_seal(n, S, w.keep)
            plan.append((c, seal))
        return plan
    while n < n0:
        c = min(chunk_max, n0 - n)
        if w.seal_trigger > 0:
            c = min(c, max(1, S + w.seal_trigger - n))
        elif w.seal_trigger == 0:
            c = min(c, w.ring - journal_len(n, S))
        n += c
        seal = should_seal(w, n, S)
        if seal:
            S += 128 * groups_to_seal(n, S, w.keep)
        plan.append((c, seal))
    return plan


def build_state(w: Workload, cache: KVCache, ds: DeviceSynth, seq_ids, layers, contexts=None, stream=0,
                chunk_max=4096):
    """Append and seal each listed sequence of each listed layer up to its context."""
    torch = ds.torch
    contexts = contexts or [w.contexts[i] for i in range(len(seq_ids))]
    buf_k = torch.empty(chunk_max * w.n_kv_heads * w.head_dim, dtype=torch.float16, device=ds.dev)
    buf_v = torch.empty_like(buf_k)
    for layer in layers:
        for seq, n0 in zip(seq_ids, contexts):
            pos = cache.state(layer, seq)[0]
            for c, seal in prefill_plan(w, n0, chunk_max):
                ds.kv(synth.T_K, layer, seq, pos, c, buf_k, stream)
                ds.kv(synth.T_V, layer, seq, pos, c, buf_v, stream)
                k = buf_k[: c * w.n_kv_heads * w.head_dim].view(1, c, w.n_kv_heads, w.head_dim)
                v = buf_v[: c * w.n_kv_heads * w.head_dim].view(1, c, w.n_kv_heads, w.head_dim)
                cache.append(layer, [seq], k, v, stream)
                pos += c
                if seal:
                    cache.seal(layer, [seq], w.keep, stream)


class DecodeInputs:
    """Per-step q / k / v of every layer, generated into HBM ahead of the timed region."""

    def __init__(self, w: Workload, ds: DeviceSynth, seq_ids, contexts, steps, layers):
        torch = ds.torch
        L = len(layers)
        B = len(seq_ids)
        H, D, Hq = w.n_kv_heads, w.head_dim, w.n_q_heads
        self.q = torch.empty((steps, L, B, Hq, D), dtype=torch.float16, device=ds.dev)
        self.k = torch.empty((steps, L, B, 1, H, D), dtype=torch.float16, device=ds.dev)
        self.v = torch.empty_like(self.k)
        for s in range(steps):
            for li, layer in enumerate(layers):
                for b, (seq, n0) in enumerate(zip(seq_ids, contexts)):
                    ds.q(layer, seq, s, self.q[s, li, b])
                    ds.kv(synth.T_K, layer, seq, n0 + s, 1, self.k[s, li, b])
                    ds.kv(synth.T_V, layer, seq, n0 + s, 1, self.v[s, li, b])


def decode_step(w: Workload, cache: KVCache, inp: DecodeInputs, step, seq_ids, layers, out, stream=0,
                on_attn=None):
    """One decode step over all layers: append, seal per policy, attention.

    out: fp16 CUDA tensor [L, B, Hq, D]. ``on_attn(layer_index, start)`` is called just before
    (start=True) and after (start=False) each attention launch (for event timing).
    Returns the number of (layer, sequence) groups sealed.
    """
    sealed = 0
    for li, layer in enumerate(layers):
        cache.append(layer, seq_ids, inp.k[step, li], inp.v[step, li], stream)
        need = []
        for seq in seq_ids:
            n, S = cache.state(layer, seq)
            if should_seal(w, n, S):
                need.append(seq)
        if need:
            sealed += cache.seal(layer, need, w.keep, stream)
        if on_attn:
            on_attn(li, True)
        cache.decode_attn(layer, seq_ids, inp.q[step, li], out[li], stream)
        if on_attn:
            on_attn(li, False)
    return sealed
