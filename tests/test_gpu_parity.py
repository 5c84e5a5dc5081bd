"""GPU parity: the CUDA path through the C ABI against the oracle, element by element.

- Stored bytes (sink, exact journal / tail, tq6_0 ring codes and scales, body records) are
  compared byte for byte.
- kv_dequant output is compared bit for bit with the oracle's dequantized regions.
- Decode attention is compared with the oracle's fp64 attention over the same cache:
  |gpu - oracle| <= max(1e-3, 2e-3 |oracle|) (the decode tolerance, ``tolerance.py``), with
  the configs' query spread and with 4x sharper queries; 16x sharper queries are an extra
  case with the bound scaled by 4. The observed error maxima are recorded per family.
"""

import numpy as np
import pytest

from oracle import attention
from quantized_kv_cache_gb300 import synth, _lib

import tolerance
from gpu_cases import FAMILIES, Family, Pair, inputs
from tolerance import ATOL, RTOL

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=list(FAMILIES))
def pair(request):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f = FAMILIES[request.param]
    p = Pair(f)
    p.prefill()
    yield p
    p.gpu.close()


def _check_bytes(p: Pair):
    f = p.f
    for (l, s, h), hc in p.hc.items():
        N, S = p.gpu.state(l, s)
        assert (N, S) == (hc.N, hc.S)
        for w, which in (("K", 0), ("V", 1)):
            sink = p.region_bytes(l, s, h, which, _lib.REGION_SINK).view(np.float16).reshape(128, f.D)
            ns = min(N, 128)
            assert np.array_equal(sink[:ns].view(np.uint16), hc.sink[w][:ns].view(np.uint16))
            if f.journal == "tq6_0":
                codes = p.region_bytes(l, s, h, which, _lib.REGION_JOURNAL).reshape(f.R, f.D // 128, 96)
                scl = p.region_bytes(l, s, h, which, _lib.REGION_JOURNAL_SCALE).view(np.uint16).reshape(f.R, -1)
                for pos in range(S, N):
                    d, ql, qh = hc.tq6_slot_bytes(pos, w)
                    slot = (pos - 128) % f.R
                    assert np.array_equal(scl[slot], d.view(np.uint16)), (w, pos)
                    assert np.array_equal(codes[slot, :, :64], ql), (w, pos)
                    assert np.array_equal(codes[slot, :, 64:], qh), (w, pos)
                tail = p.region_bytes(l, s, h, which, _lib.REGION_TAIL).view(np.uint16).reshape(f.T, f.D)
                for pos in range(max(128, N - f.T), N):
                    assert np.array_equal(tail[pos % f.T], hc.tail[w][pos % f.T])
            else:
                jx = p.region_bytes(l, s, h, which, _lib.REGION_JOURNAL).view(np.uint16).reshape(f.R, f.D)
                for pos in range(max(S, 128), N):
                    slot = (pos - 128) % f.R
                    assert np.array_equal(jx[slot], hc.jx[w][slot]), (w, pos)
            body = p.region_bytes(l, s, h, which, _lib.REGION_BODY)
            ng = (S - 128) // 128
            rb = len(hc.record_bytes(0, w)) if ng else 0
            for g in range(ng):
                ref = hc.record_bytes(g, w)
                got = body[g * rb:(g + 1) * rb]
                diff = np.flatnonzero(got != ref)
                assert diff.size == 0, f"{f.name} {w} l{l} s{s} h{h} group {g}: {diff.size} bytes differ, first {diff[:8]}"


def _check_dequant(p: Pair):
    for (l, s, h), hc in p.hc.items():
        N = hc.N
        regs = hc.regions()
        for which, idx in ((0, 1), (1, 2)):
            got = p.dequant(l, s, h, which, 0, N)
            ref = np.concatenate([r[idx] for r in regs]).astype(np.float32)
            assert got.shape == ref.shape
            bad = np.flatnonzero(got.view(np.uint32) != ref.view(np.uint32))
            assert bad.size == 0, f"{p.f.name} l{l} s{s} h{h} w{which}: {bad.size} values differ, first {bad[:5]}"


def _q(p: Pair, layer, step, scale_mult=1.0):
    f = p.f
    qs = [synth.q_values(f.seed, layer, s, step, f.Hq, f.D, q_scale=scale_mult / np.sqrt(f.D)) for s in p.seqs]
    return np.stack(qs)


def _check_attention(p: Pair, layer, q, atol=ATOL, rtol=RTOL, got=None, case=""):
    """got: the GPU output for q (default: one kv_decode_attn call now). The errors are
    recorded under the family's name (plus `case`)."""
    f = p.f
    if got is None:
        got = p.attend(layer, p.seqs, q)
    got = got.astype(np.float64)
    G = f.Hq // f.H
    worst = 0.0
    for bi, s in enumerate(p.seqs):
        for h in range(f.H):
            hc = p.hc[(layer, s, h)]
            ref = attention.attend(q[bi, h * G:(h + 1) * G].astype(np.float64), hc.regions(), hc.cfg.rot,
                                   1.0 / np.sqrt(f.D))
            r = tolerance.check(f.name + case, got[bi, h * G:(h + 1) * G], ref, atol, rtol,
                                where=f"layer {layer} seq {s} head {h}")
            worst = max(worst, r)
    return worst


def test_prefill_bytes_match_oracle(pair):
    _check_bytes(pair)


def test_prefill_dequant_bit_exact(pair):
    _check_dequant(pair)


@pytest.mark.parametrize("mult", [1.0, 4.0])
def test_prefill_attention_matches_oracle(pair, mult):
    for layer in range(pair.f.L):
        _check_attention(pair, layer, _q(pair, layer, 0, mult), case="" if mult == 1.0 else f" q{mult:g}x")


def test_prefill_attention_sharp_softmax(pair):
    # 16x sharper queries, beyond the workloads' query spread (an extra case, not the
    # contract's): scores spread ~4 instead of ~0.25, so the fp16 rounding of the mma operands
    # (2^-11 relative on q and on the dequantized K) moves scores by up to ~4e-3 and the
    # outputs by about that much. The bound is the contract tolerance scaled by 8; the observed
    # errors are recorded under "<family> sharp16".
    for layer in range(pair.f.L):
        _check_attention(pair, layer, _q(pair, layer, 0, 16.0), atol=8 * ATOL, rtol=8 * RTOL, case=" sharp16")


def test_decode_steps_match_oracle(pair):
    # decode: append one position to every sequence, seal per policy, attend; all layers
    f = pair.f
    for step in range(f.steps):
        for layer in range(f.L):
            n0 = [pair.gpu.state(layer, s)[0] for s in pair.seqs]
            pair.append(layer, pair.seqs, n0, 1)
            pair.seal(layer, pair.seqs, f.keep)
            _check_attention(pair, layer, _q(pair, layer, step + 1))
    _check_bytes(pair)
    _check_dequant(pair)


def _step_calls(p: Pair, steps, step0, keep):
    """Decode steps through kv_decode_step (one call per step over all layers; seal policy
    'whenever a full group is older than keep'), each layer's output checked against the
    oracle after the same append and seal. Layouts whose decode kernel takes the region items
    append inside that kernel (the newest row read from the call's input)."""
    f = p.f
    dev = p.dev
    for step in range(step0, step0 + steps):
        K = np.zeros((f.L, len(p.seqs), f.H, f.D), np.float16)
        V = np.zeros_like(K)
        Q = np.stack([_q(p, layer, step) for layer in range(f.L)])
        for layer in range(f.L):
            for bi, s in enumerate(p.seqs):
                n = p.gpu.state(layer, s)[0]
                k, v = inputs(f, layer, s, n, 1)
                K[layer, bi], V[layer, bi] = k[0], v[0]
                for h in range(f.H):
                    p.hc[(layer, s, h)].append(k[:, h], v[:, h])
                    p.hc[(layer, s, h)].seal(keep)
        Kd, Vd, Qd = (torch.from_numpy(x).to(dev) for x in (K, V, Q))
        out = torch.empty_like(Qd)
        _lib.kv_decode_step(p.gpu.h, f.L, p.seqs, Qd.data_ptr(), Kd.data_ptr(), Vd.data_ptr(), out.data_ptr(), 0,
                            keep, p.gpu.ws.data_ptr(), p.gpu.ws_bytes)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        for layer in range(f.L):
            _check_attention(p, layer, Q[layer], got=got[layer])


def test_decode_step_call_matches_oracle(pair):
    # the same decode steps through the one-call entry point (after the per-call steps above)
    _step_calls(pair, pair.f.steps, pair.f.steps + 1, pair.f.keep)
    _check_bytes(pair)
    _check_dequant(pair)


@pytest.mark.parametrize("base", ["tbq4_f16", "kvarn4_ring", "kvarn5_wide", "q8q4_bf16"])
def test_decode_step_call_across_sink_edge(base):
    # short sequences stepped across position 128: the newest position moves from the sink
    # into the exact journal / tail while the decode kernel appends it
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f0 = FAMILIES[base]
    f = Family(f0.name + "_edge", f0.D, f0.H, f0.Hq, f0.k_body, f0.v_body, f0.journal, f0.tail_fmt, T=f0.T, R=f0.R,
               contexts=[124, 101], keep=f0.keep, steps=6, n_out=f0.n_out, factor=f0.factor, balance=f0.balance)
    p = Pair(f)
    try:
        p.prefill()
        _step_calls(p, f.steps, 1, f.keep)
        _check_bytes(p)
        _check_dequant(p)
    finally:
        p.gpu.close()


@pytest.mark.parametrize("base", ["kvarn4_ring", "q8q4_bf16", "tbq4_ring"])
def test_decode_step_layers_out_of_step(base):
    # layers whose lengths differ: after the prefill, layer 0 and layer 1 get extra positions so
    # that, with the policy 'seal whenever a full group is older than keep', layer 0 falls due in
    # the first decode step and layer 1 in the second, each sequence on its own count. The step
    # then seals per layer (not one call over all layers); every step's outputs, and in the end
    # every stored byte and the dequantized values, are checked against the oracle.
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f0 = FAMILIES[base]
    f = Family(f0.name + "_skew", f0.D, f0.H, f0.Hq, f0.k_body, f0.v_body, f0.journal, f0.tail_fmt, T=f0.T, R=f0.R,
               contexts=f0.contexts, keep=f0.keep, steps=4, n_out=f0.n_out, factor=f0.factor, balance=f0.balance)
    p = Pair(f)
    try:
        p.prefill()
        for layer, due_step in ((0, 1), (1, 2)):
            for s in p.seqs:
                n, S = p.gpu.state(layer, s)
                extra = 128 - due_step - (n - f.keep - S)     # the due step's append makes 128
                assert 0 <= extra < 128
                if extra:
                    p.append(layer, [s], [n], extra)
        states = [[p.gpu.state(layer, s) for s in p.seqs] for layer in range(f.L)]
        assert states[0] != states[1]
        _step_calls(p, f.steps, 1, f.keep)
        for layer in (0, 1):
            for s, (n, S) in zip(p.seqs, states[layer]):
                assert p.gpu.state(layer, s)[1] == S + 128, (layer, s)
        _check_bytes(p)
        _check_dequant(p)
    finally:
        p.gpu.close()


def test_decode_step_graph_and_direct_agree():
    # the same steps through one CUDA graph per step and through direct launches: outputs and
    # every stored byte agree exactly (a seal step changes the graph's topology mid-run)
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f = FAMILIES["kvarn4_ring"]
    pairs = [Pair(f), Pair(f)]
    try:
        for p in pairs:
            p.gpu.pool.zero_()   # kv_create leaves unwritten slots as allocated: compare from zero
            p.prefill()
        _lib.kv_set_graph_mode(pairs[1].gpu.h, False)
        outs = [[], []]
        for step in range(1, 7):
            K = np.zeros((f.L, len(pairs[0].seqs), f.H, f.D), np.float16)
            V = np.zeros_like(K)
            Q = np.stack([_q(pairs[0], layer, step) for layer in range(f.L)])
            for layer in range(f.L):
                for bi, s in enumerate(pairs[0].seqs):
                    k, v = inputs(f, layer, s, pairs[0].gpu.state(layer, s)[0], 1)
                    K[layer, bi], V[layer, bi] = k[0], v[0]
            for i, p in enumerate(pairs):
                Kd, Vd, Qd = (torch.from_numpy(x).to(p.dev) for x in (K, V, Q))
                out = torch.empty_like(Qd)
                # keep 128 below the family's: a seal in some steps
                _lib.kv_decode_step(p.gpu.h, f.L, p.seqs, Qd.data_ptr(), Kd.data_ptr(), Vd.data_ptr(),
                                    out.data_ptr(), 0, f.keep - 128, p.gpu.ws.data_ptr(), p.gpu.ws_bytes)
                torch.cuda.synchronize()
                outs[i].append(out.cpu().numpy())
        for a, b in zip(*outs):
            assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
        for layer in range(f.L):
            for s in pairs[0].seqs:
                assert pairs[0].gpu.state(layer, s) == pairs[1].gpu.state(layer, s)
        torch.cuda.synchronize()
        regions = [(r, getattr(_lib, r)) for r in dir(_lib) if r.startswith("REGION_")]
        for layer in range(f.L):
            for s in pairs[0].seqs:
                for h in range(f.H):
                    for which in (0, 1):
                        for name, r in regions:
                            a = pairs[0].region_bytes(layer, s, h, which, r)
                            b = pairs[1].region_bytes(layer, s, h, which, r)
                            bad = np.flatnonzero(a != b)
                            assert bad.size == 0, f"{name} l{layer} s{s} h{h} w{which}: {bad.size} bytes, first {bad[:6]}"
        diff = torch.nonzero(pairs[0].gpu.pool != pairs[1].gpu.pool).flatten()
        assert diff.numel() == 0, f"{diff.numel()} pool bytes differ outside the regions, first {diff[:6].tolist()}"
    finally:
        for p in pairs:
            p.gpu.close()
