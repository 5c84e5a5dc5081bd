"""GPU parity on the edge cases of the codec and of the decode work list.

- Degenerate values (every format family): 128-position groups that are all zero, constant,
  alternating +-c, fp16 subnormals, large (scales still finite), or one dominant channel per row,
  between groups of the seeded normal values. These reach the codecs' special cases: a zero
  TBQ4 norm, a zero Q8_0 / Q4_0 scale, KVarN rows and columns whose spread is 0 (counted as
  1) and tiles whose rows have no range, tq6_0 scales that underflow. Stored bytes and
  dequantized values must equal the oracle's exactly, and the status word stays clear.
- fp16 scale overflow (TBQ4): rows whose 128-value norm exceeds the fp16 maximum give the same
  (infinite) stored norms and the same codes as the oracle, and the encoder flags them in bit 0
  of the status word. (KVarN's balancing splits a row's magnitude between its row and column
  scales, so the same inputs leave its fp16 scales finite.)
- Ragged lengths: sequences of 1, 127, 128, 129, 256, 257 and 600 positions in one cache and one
  call (sink only, the sink's last position, the first journal position, group boundaries),
  including groups of zeros and constants, through decode steps; attention within the decode
  tolerance.
- The per-call maximum: 32 sequences in one kv_decode_attn / kv_decode_step call.
"""

import numpy as np
import pytest

from oracle.cache import HeadCache
from quantized_kv_cache_gb300 import synth, _lib

from gpu_cases import FAMILIES, Family, Pair, inputs
from test_gpu_parity import _check_attention, _check_bytes, _check_dequant, _q, _step_calls

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

PATTERNS = ["normal", "zero", "const", "alt", "subnormal", "huge", "spike"]


def special_rows(kind, n, H, D, seed):
    """fp16 [n, H, D] rows of one pattern (deterministic; 'normal' from the seeded streams)."""
    rng = np.random.default_rng(seed)
    if kind == "zero":
        return np.zeros((n, H, D), np.float16)
    if kind == "const":
        return np.full((n, H, D), 0.75, np.float16)
    if kind == "alt":
        x = np.ones((n, H, D), np.float32) * 1.5
        x[..., 1::2] = -1.5
        return x.astype(np.float16)
    if kind == "subnormal":
        return (rng.standard_normal((n, H, D)) * 3e-7).astype(np.float16)
    if kind == "huge":        # large values whose fp16 scales still fit (a TBQ4 norm ~2,000 x sqrt(128))
        return np.clip(rng.standard_normal((n, H, D)) * 2000.0, -65000, 65000).astype(np.float16)
    if kind == "overflow":    # a TBQ4 norm (~20,000 x sqrt(128)) beyond the fp16 maximum
        return np.clip(rng.standard_normal((n, H, D)) * 20000.0, -65000, 65000).astype(np.float16)
    if kind == "spike":
        x = rng.standard_normal((n, H, D)) * 0.01
        x[..., 5] = 300.0
        return x.astype(np.float16)
    raise ValueError(kind)


class EdgePair(Pair):
    """A Pair whose positions take a pattern per 128-position group (group index g of the
    journal, counted from position 128; the sink takes the seeded values)."""

    def __init__(self, f, patterns, device=0):
        super().__init__(f, device)
        self.patterns = patterns

    def rows(self, layer, seq, pos0, n):
        f = self.f
        k, v = inputs(f, layer, seq, pos0, n)
        k, v = k.copy(), v.copy()
        for i in range(n):
            pos = pos0 + i
            if pos < 128:
                continue
            kind = self.patterns[((pos - 128) // 128) % len(self.patterns)]
            if kind != "normal":
                seed = 1000 * layer + 100 * seq + (pos - 128) // 128
                k[i] = special_rows(kind, 1, f.H, f.D, seed)[0]
                v[i] = special_rows(kind, 1, f.H, f.D, seed + 7)[0]
        return k, v

    def append(self, layer, seqs, pos0s, n):
        ks, vs = [], []
        for s, p0 in zip(seqs, pos0s):
            k, v = self.rows(layer, s, p0, n)
            ks.append(k)
            vs.append(v)
            for h in range(self.f.H):
                self.hc[(layer, s, h)].append(k[:, h], v[:, h])
        K = self.torch.from_numpy(np.stack(ks)).to(self.dev)
        V = self.torch.from_numpy(np.stack(vs)).to(self.dev)
        self.gpu.append(layer, seqs, K, V)


def _fill(p, chunk=200):
    """Append every sequence of every layer up to its context in chunks, sealing after each."""
    f = p.f
    for layer in range(f.L):
        for s, n0 in zip(p.seqs, f.contexts):
            pos = 0
            while pos < n0:
                N, S = p.gpu.state(layer, s)
                c = min(chunk, n0 - pos, f.R - (max(N, 128) - S))
                p.append(layer, [s], [pos], c)
                pos += c
                p.seal(layer, [s], f.keep)


@pytest.mark.parametrize("name", list(FAMILIES))
def test_degenerate_values_bytes_and_dequant(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f0 = FAMILIES[name]
    n_groups = len(PATTERNS) + 1
    ctx = 128 + 128 * n_groups + f0.keep + 50
    f = Family(f0.name + "_deg", f0.D, f0.H, f0.Hq, f0.k_body, f0.v_body, f0.journal, f0.tail_fmt, T=f0.T,
               R=f0.R, contexts=[ctx], keep=f0.keep, steps=0, L=1, seed=f0.seed + 5, n_out=f0.n_out,
               factor=f0.factor, balance=f0.balance)
    p = EdgePair(f, PATTERNS)
    try:
        _fill(p)
        assert p.gpu.state(0, 0)[1] >= 128 + 128 * len(PATTERNS)   # every pattern sealed
        assert _lib.kv_get_status(p.gpu.h) == 0
        _check_bytes(p)
        _check_dequant(p)
    finally:
        p.gpu.close()


@pytest.mark.parametrize("name", ["tbq4_ring", "kvarn4_ring", "q8q4_bf16", "kvarn5_wide"])
def test_ragged_lengths_attention(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f0 = FAMILIES[name]
    contexts = [1, 127, 128, 129, 256, 257, 600]
    f = Family(f0.name + "_rag", f0.D, f0.H, f0.Hq, f0.k_body, f0.v_body, f0.journal, f0.tail_fmt, T=f0.T,
               R=f0.R, contexts=contexts, keep=f0.keep, steps=2, L=1, seed=f0.seed + 11, n_out=f0.n_out,
               factor=f0.factor, balance=f0.balance)
    p = EdgePair(f, ["normal", "zero", "const", "normal"])
    try:
        _fill(p, chunk=97)
        for mult in (1.0, 4.0):
            _check_attention(p, 0, _q(p, 0, 0, mult), case=f" edges q{mult:g}x")
        _step_calls(p, f.steps, 1, f.keep)      # kv_decode_step over all seven sequences
        _check_bytes(p)
    finally:
        p.gpu.close()


def test_thirty_two_sequences_in_one_call():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f0 = FAMILIES["tbq4_ring"]
    contexts = [100 + 61 * i for i in range(32)]
    f = Family("tbq4_ring_32", f0.D, f0.H, f0.Hq, f0.k_body, f0.v_body, f0.journal, f0.tail_fmt, T=f0.T,
               R=f0.R, contexts=contexts, keep=f0.keep, steps=1, L=1, seed=21, n_out=f0.n_out, factor=f0.factor, balance=f0.balance)
    p = Pair(f)
    try:
        for s, n0 in zip(p.seqs, f.contexts):
            pos = 0
            while pos < n0:
                N, S = p.gpu.state(0, s)
                c = min(300, n0 - pos, f.R - (max(N, 128) - S))
                p.append(0, [s], [pos], c)
                pos += c
                p.seal(0, [s], f.keep)
        assert len(p.seqs) == 32
        _check_attention(p, 0, _q(p, 0, 0), case=" edges")
        _step_calls(p, 1, 1, f.keep)
        _check_bytes(p)
    finally:
        p.gpu.close()


@pytest.mark.parametrize("name", ["tbq4_f16", "tbq4_ring"])
def test_fp16_scale_overflow_is_flagged(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f0 = FAMILIES[name]
    ctx = 128 + 128 * 2 + f0.keep + 10
    f = Family(f0.name + "_ovf", f0.D, f0.H, f0.Hq, f0.k_body, f0.v_body, f0.journal, f0.tail_fmt, T=f0.T,
               R=f0.R, contexts=[ctx], keep=f0.keep, steps=0, L=1, seed=f0.seed + 17, n_out=f0.n_out,
               factor=f0.factor, balance=f0.balance)
    p = EdgePair(f, ["normal", "overflow"])
    try:
        _fill(p)
        assert p.gpu.state(0, 0)[1] >= 128 + 2 * 128
        assert _lib.kv_get_status(p.gpu.h) & 1
        _check_bytes(p)    # the stored bytes, infinite scales included, are the oracle's
    finally:
        p.gpu.close()


def test_bounded_wait_runs_out_and_sets_status_bit1():
    """The streaming kernels' bounded wait: a test launch waits 1 ms on an mbarrier that no copy
    completes; the wait gives up, bit 1 of the status word is set (kv_get_status reports
    KVQ_EDEVICE), the launch retires, and the same context then decodes correctly."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f = FAMILIES["tbq4_ring"]
    p = Pair(f)
    try:
        p.prefill()
        assert _lib.kv_get_status(p.gpu.h) == 0
        _lib.kv_test_wait_timeout(p.gpu.h, 1_000_000)
        torch.cuda.synchronize()
        code = _lib.load().kv_get_status(p.gpu.h, None)
        assert code == 5                                   # KVQ_EDEVICE, and the word is cleared
        assert _lib.kv_get_status(p.gpu.h) == 0
        _lib.kv_test_wait_timeout(p.gpu.h, 1_000_000)
        torch.cuda.synchronize()
        assert _lib.kv_get_status(p.gpu.h) == 2            # bit 1 alone
        with pytest.raises(_lib.KVQError):
            _lib.kv_test_wait_timeout(p.gpu.h, 10)        # limit out of range
        _check_attention(p, 0, _q(p, 0, 0), case=" after wait timeout")
        assert _lib.kv_get_status(p.gpu.h) == 0
    finally:
        p.gpu.close()
