"""GPU parity of kv_prefill, the bulk prefill with groups sealed straight from the chunk.

kv_prefill must leave the cache byte for byte as kv_append of the chunk followed by kv_seal(keep)
would, although it writes a group that the call seals straight from the input rows (through the
values the journal would hold) and therefore takes chunks far larger than the journal ring. The
oracle reaches the same state the plain way: appends of journal-sized pieces, each followed by
seal(keep) (a record depends only on its group's rows, not on when it is sealed). Checked on
every format family: a first chunk inside the sink, a second that finishes the sink and holds
whole groups, a third that starts inside a group (its head completes a group already in the
journal, sealed from there), and a short fourth one that seals nothing; every stored region byte for byte, dequant bit for bit, and
attention within the decode tolerance; the refusals on the host.
"""

import numpy as np
import pytest

from quantized_kv_cache_gb300 import _lib

from gpu_cases import FAMILIES, Family, Pair, inputs
from test_gpu_parity import _check_attention, _check_bytes, _check_dequant, _q

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


class PrefillPair(Pair):
    def prefill_call(self, layer, n):
        """One kv_prefill of n positions for every sequence; the oracle's plain replay."""
        f = self.f
        ks, vs = [], []
        for s in self.seqs:
            N0 = self.gpu.state(layer, s)[0]
            k, v = inputs(f, layer, s, N0, n)
            ks.append(k)
            vs.append(v)
            for h in range(f.H):
                hc = self.hc[(layer, s, h)]
                done = 0
                while done < n:
                    room = f.R - (max(hc.N, 128) - hc.S)
                    c = min(n - done, room)
                    assert c > 0
                    hc.append(k[done:done + c, h], v[done:done + c, h])
                    hc.seal(f.keep)
                    done += c
        K = torch.from_numpy(np.ascontiguousarray(np.stack(ks))).to(self.dev)
        V = torch.from_numpy(np.ascontiguousarray(np.stack(vs))).to(self.dev)
        g = _lib.kv_prefill(self.gpu.h, layer, self.seqs, n, K.data_ptr(), V.data_ptr(), f.keep)
        torch.cuda.synchronize()
        return g


@pytest.mark.parametrize("name", list(FAMILIES))
def test_prefill_matches_append_then_seal(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f0 = FAMILIES[name]
    # chunks: 60 sink positions; up to 3.3 rings (the sink's rest, whole groups straight from the
    # input); 2 rings + 71 starting inside a group; 40 positions that seal nothing
    n1 = int(3.3 * f0.R)
    chunks = (60, n1 - 60, 2 * f0.R + 71, 40)
    f = Family(f0.name + "_pf", f0.D, f0.H, f0.Hq, f0.k_body, f0.v_body, f0.journal, f0.tail_fmt, T=f0.T,
               R=f0.R, contexts=[sum(chunks)] * 2, keep=f0.keep, steps=0, L=2, seed=f0.seed + 23,
               n_out=f0.n_out, factor=f0.factor, balance=f0.balance)
    p = PrefillPair(f)
    try:
        for layer in range(f.L):
            for n in chunks:
                before = [p.gpu.state(layer, s)[1] for s in p.seqs]
                g = p.prefill_call(layer, n)
                after = [p.gpu.state(layer, s)[1] for s in p.seqs]
                assert g == sum((a - b) // 128 for a, b in zip(after, before))
                for s in p.seqs:
                    hc = p.hc[(layer, s, 0)]
                    assert p.gpu.state(layer, s) == (hc.N, hc.S)
        assert _lib.kv_get_status(p.gpu.h) == 0
        _check_bytes(p)
        _check_dequant(p)
        for layer in range(f.L):
            _check_attention(p, layer, _q(p, layer, 0), case=" prefill")
    finally:
        p.gpu.close()


def test_prefill_refusals():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f0 = FAMILIES["tbq4_ring"]
    f = Family("pf_refuse", f0.D, f0.H, f0.Hq, f0.k_body, f0.v_body, f0.journal, f0.tail_fmt, T=f0.T, R=f0.R,
               contexts=[5000], keep=f0.keep, steps=0, L=1, seed=3, balance=f0.balance)
    p = PrefillPair(f)
    try:
        H, D = f.H, f.D
        big = torch.zeros((1, p.gpu.cfg.max_ctx + 1, H, D), dtype=torch.float16, device=p.dev)
        with pytest.raises(_lib.KVQError) as e:      # beyond max_ctx
            _lib.kv_prefill(p.gpu.h, 0, [0], p.gpu.cfg.max_ctx + 1, big.data_ptr(), big.data_ptr(), f.keep)
        assert "ENOSPC" in str(e.value)
        x = torch.zeros((1, 4 * f.R, H, D), dtype=torch.float16, device=p.dev)
        with pytest.raises(_lib.KVQError) as e:      # keep so large that the unsealed rest overflows the ring
            _lib.kv_prefill(p.gpu.h, 0, [0], 4 * f.R, x.data_ptr(), x.data_ptr(), 2 * f.R)
        assert "ENOSPC" in str(e.value)
        with pytest.raises(_lib.KVQError):           # keep below the tail
            _lib.kv_prefill(p.gpu.h, 0, [0], 10, x.data_ptr(), x.data_ptr(), f.T - 1)
        assert p.gpu.state(0, 0) == (0, 128)         # nothing written
    finally:
        p.gpu.close()
