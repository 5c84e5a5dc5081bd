"""GPU parity at the workloads' full sizes, in the launch configuration the bench times.

The five configured workloads run with every layer allocated (fa14b's 48-layer pool is about
10 GB, longctx's 16-layer pool about 18 GB, so the later layers' storage lies beyond 2 GiB of
pool offset) and every decode step of their recipe:

- the cache is built the way ``bench.py`` builds it: the device-side seeded generator fills
  the rows and the bench's prefill plan appends and seals them, for all layers;
- every decode step goes through ``kv_decode_step`` (one CUDA graph per step: append, seal by
  the workload's policy, decode attention and merge over all layers); hybrid27b's journal
  reaches its 8,192 mark at step 128 and seals 32 groups per layer inside the step; longctx
  runs its bulk seal of 4 x 128 groups per layer (one kv_seal over all layers) after step 16.

For sampled (sequence, KV head) pairs on layers {0, L/2, L-1} the oracle replays the same
appends and seals from the host-side generator (the same counter-based streams) and the
test compares, after the last step:

- the sequence's lengths (N, S) and the groups each step sealed;
- every body record of the sampled heads (K and V), byte for byte, the step's seals included;
- every journal row of the unsealed span (tq6_0 codes and scales, or exact rows) and every
  exact-tail row;
- kv_dequant over all N positions (every region) bit for bit against the oracle's dequantized
  regions;
- the decode output of the head's query group at the first and at the last step against the
  fp64 oracle attention, within max(1e-3, 2e-3 |oracle|) (``tolerance.py``).

The three workloads of the widened rows (KVarN 3/2, q5_1 / q4_0, tq5_0 / TBQ4) run one layer
and one step with the same checks. The bench's prefill measurement (kv_prefill of a sampled
sequence's whole context into a fresh one-layer cache) is checked as well: lengths, every
sealed record and the newest journal and tail rows.
"""

import copy
import dataclasses

import numpy as np
import pytest

import tolerance
from oracle import attention, codecs
from oracle.cache import HeadCache, HeadConfig
from quantized_kv_cache_gb300 import configs, synth, _lib

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

# workload -> sampled (sequence, KV head) pairs; these run every layer and every step
FULL = {
    "tiny_tbq4": [(0, 0), (0, 1)],
    "hybrid27b_kvarn44": [(0, 3)],
    "fa14b_q8q4": [(0, 5)],
    "widehead_kvarn55": [(2, 1), (7, 0)],
    "longctx_tbq4": [(0, 2), (3, 0)],
}
# the widened rows' workloads: one layer, one step
ONE_LAYER = {
    "hybrid27b_kvarn32_200k": [(0, 2)],
    "fa14b_q51q40": [(0, 3)],
    "hybrid27b_tq50tbq4_110k": [(0, 1)],
}


def _step_trigger(w):
    """Seal trigger of the decode step: tiny_tbq4's recipe seals its 6 groups in the step
    (after the append, before the attention); the other workloads follow their policy."""
    return 0 if w.seal_trigger == -1 else w.seal_trigger


def _layers(w):
    return sorted({0, w.n_layers // 2, w.n_layers - 1})


class Run:
    pass


def _gpu_run(w, steps):
    """Builds the workload's cache on the device as the bench does and runs `steps` decode
    steps through kv_decode_step. Keeps the outputs of the first and the last step."""
    from quantized_kv_cache_gb300 import KVCache
    from quantized_kv_cache_gb300.runner import DeviceSynth, DecodeInputs, build_state
    dev = torch.device("cuda", 0)
    cfg = w.config()
    cfg.max_ctx = max(w.contexts) + max(steps, w.steps) + 512 + 32 * 128     # as bench.py sizes it
    cache = KVCache(cfg, 0)
    ds = DeviceSynth(w, 0)
    seq_ids = list(range(len(w.contexts)))
    stream = torch.cuda.current_stream(dev).cuda_stream
    layers = list(range(w.n_layers))
    build_state(w, cache, ds, seq_ids, layers, stream=stream)
    inp = DecodeInputs(w, ds, seq_ids, w.contexts, steps, layers)
    out = torch.empty((w.n_layers, len(seq_ids), w.n_q_heads, w.head_dim), dtype=torch.float16, device=dev)
    r = Run()
    r.sealed, r.bulk = [], 0
    for s in range(steps):
        if w.bulk_seal_step >= 0 and s == w.bulk_seal_step:
            r.bulk = _lib.kv_seal(cache.h, -1, seq_ids, w.keep, stream)
        r.sealed.append(_lib.kv_decode_step(cache.h, w.n_layers, seq_ids, inp.q[s].data_ptr(), inp.k[s].data_ptr(),
                                            inp.v[s].data_ptr(), out.data_ptr(), _step_trigger(w), w.keep,
                                            cache.ws.data_ptr(), cache.ws_bytes, None, stream))
        if s == 0:
            torch.cuda.synchronize()
            r.first = out.cpu().numpy()
    torch.cuda.synchronize()
    r.last = out.cpu().numpy()
    r.status = _lib.kv_get_status(cache.h)
    r.w, r.cache, r.inp, r.steps = w, cache, inp, steps
    del inp
    return r


def _rows(w, layer, seq, h, p0, n):
    k = synth.kv_values(w.seed, synth.T_K, layer, seq, h, p0, n, w.head_dim, w.n_out, w.out_factor)
    v = synth.kv_values(w.seed, synth.T_V, layer, seq, h, p0, n, w.head_dim)
    return k, v


def _replay(w, layer, seq, h, steps):
    """The oracle's cache of (layer, seq, h) replayed through the bench's prefill and `steps`
    decode steps, the attention references of the first and the last step, the groups each
    step sealed, and a copy of the cache right after the prefill."""
    from quantized_kv_cache_gb300.runner import prefill_plan
    D, G = w.head_dim, w.G
    hc = HeadCache(HeadConfig(D, w.k_body, w.v_body, w.journal, w.tail_fmt, w.tail, w.ring))
    n0 = w.contexts[seq]
    pos = 0
    for c, seal in prefill_plan(w, n0):
        hc.append(*_rows(w, layer, seq, h, pos, c))
        pos += c
        if seal:
            hc.seal(w.keep)
    after_prefill = copy.deepcopy(hc) if layer == 0 else None
    trig = dataclasses.replace(w, seal_trigger=_step_trigger(w))
    refs, sealed = {}, []
    for s in range(steps):
        if w.bulk_seal_step >= 0 and s == w.bulk_seal_step:
            hc.seal(w.keep)
        hc.append(*_rows(w, layer, seq, h, n0 + s, 1))
        sealed.append(hc.seal(w.keep) if configs.should_seal(trig, hc.N, hc.S) else 0)
        if s in (0, steps - 1):
            q = synth.q_values(w.seed, layer, seq, s, w.n_q_heads, D)[h * G:(h + 1) * G].astype(np.float64)
            refs[s] = attention.attend(q, hc.regions(), hc.cfg.rot, 1.0 / np.sqrt(D))
    return hc, refs, sealed, after_prefill


def _region(cache, layer, seq, head, which, region):
    ptr, nb = _lib.kv_region_ptr(cache.h, layer, seq, head, which, region)
    off = ptr - cache.pool.data_ptr()
    assert 0 <= off and off + nb <= cache.pool_bytes
    return cache.pool[off:off + nb].cpu().numpy(), off


def _check_body(w, hc, body, role, ng, where):
    if ng == 0:
        return
    rb = len(hc.record_bytes(0, role))
    ref = np.concatenate([hc.record_bytes(g, role) for g in range(ng)])
    got = body[:ng * rb]
    if not np.array_equal(got, ref):
        bad = np.flatnonzero(got != ref)
        raise AssertionError(f"{w.name} {where} {role}: {bad.size} record bytes differ, first in group "
                             f"{bad[0] // rb} (byte {bad[0] % rb})")


def _check_journal(w, cache, hc, layer, seq, h, which, role, positions, where):
    """Every listed position's journal row: tq6_0 codes and scales, or the exact row."""
    D = w.head_dim
    positions = np.asarray(list(positions), dtype=np.int64)
    if positions.size == 0:
        return
    slots = (positions - 128) % w.ring
    if w.journal == "tq6_0":
        codes = _region(cache, layer, seq, h, which, _lib.REGION_JOURNAL)[0].reshape(w.ring, D // 128, 96)
        sc = _region(cache, layer, seq, h, which, _lib.REGION_JOURNAL_SCALE)[0].view(np.uint16).reshape(w.ring, D // 128)
        ql, qh = codecs.tq6_pack(hc.jcode[role][slots])
        assert np.array_equal(codes[slots], np.concatenate([ql, qh], axis=-1)), f"{where} {role} ring codes"
        assert np.array_equal(sc[slots], hc.jd[role][slots].view(np.uint16)), f"{where} {role} ring scales"
    else:
        jx = _region(cache, layer, seq, h, which, _lib.REGION_JOURNAL)[0].view(np.uint16).reshape(w.ring, D)
        assert np.array_equal(jx[slots], hc.jx[role][slots]), f"{where} {role} journal rows"


def _check_tail(w, cache, hc, layer, seq, h, which, role, where):
    if w.journal != "tq6_0":
        return
    D = w.head_dim
    tail = _region(cache, layer, seq, h, which, _lib.REGION_TAIL)[0].view(np.uint16).reshape(w.tail, D)
    pos = np.arange(max(128, hc.N - w.tail), hc.N) % w.tail
    assert np.array_equal(tail[pos], hc.tail[role][pos]), f"{where} {role} exact tail"


def _check_dequant(w, cache, hc, layer, seq, h, where):
    regs = hc.regions()
    for which, idx in ((0, 1), (1, 2)):
        out = torch.empty((hc.N, w.head_dim), dtype=torch.float32, device=torch.device("cuda", 0))
        _lib.kv_dequant(cache.h, layer, seq, h, which, 0, hc.N, out.data_ptr())
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        del out
        ref = np.concatenate([r[idx] for r in regs]).astype(np.float32)
        assert got.shape == ref.shape
        bad = np.flatnonzero(got.view(np.uint32) != ref.view(np.uint32))
        assert bad.size == 0, f"{w.name} {where} which {which}: {bad.size} dequantized values differ, first {bad[:5]}"


@pytest.fixture(scope="module", params=list(FULL) + list(ONE_LAYER))
def run(request):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = configs.WORKLOADS[request.param]
    if request.param in ONE_LAYER:
        w = dataclasses.replace(w, n_layers=1)
        steps, samples = 1, ONE_LAYER[request.param]
    else:
        steps, samples = w.steps, FULL[request.param]
    r = _gpu_run(w, steps)
    r.samples = samples
    r.oracle = {}
    for layer in _layers(w):
        for seq, h in samples:
            r.oracle[(layer, seq, h)] = _replay(w, layer, seq, h, steps)
    yield r
    r.cache.close()
    torch.cuda.empty_cache()


def test_fullsize_inputs_and_status(run):
    w = run.w
    assert run.status == 0
    # the device generator draws the host generator's values (the oracle's inputs)
    for layer in _layers(w):
        for seq in range(len(w.contexts)):
            q = synth.q_values(w.seed, layer, seq, 0, w.n_q_heads, w.head_dim)
            assert np.array_equal(run.inp.q[0, layer, seq].cpu().numpy().view(np.uint16), q.view(np.uint16))
    assert np.all(np.isfinite(run.first)) and np.all(np.isfinite(run.last))


def test_fullsize_lengths_and_seals(run):
    w = run.w
    for (layer, seq, h), (hc, refs, sealed, _) in run.oracle.items():
        assert run.cache.state(layer, seq) == (hc.N, hc.S), (layer, seq, h)
    # groups each step sealed (all layers, all sequences) equal the oracle's per-head counts
    # summed over layers and sequences: every layer of a sequence follows the same lengths
    per_seq = {}
    for (layer, seq, h), (hc, refs, sealed, _) in run.oracle.items():
        per_seq.setdefault(seq, sealed)
        assert sealed == per_seq[seq]
    if len(per_seq) == len(w.contexts):
        expect = [w.n_layers * sum(per_seq[s][i] for s in per_seq) for i in range(run.steps)]
        assert run.sealed == expect
    if w.name == "hybrid27b_kvarn44":
        # the journal reaches 8,192 positions in the 128th step: one seal of 32 groups per layer
        assert run.sealed[127] == 32 * w.n_layers and sum(run.sealed) == 32 * w.n_layers
    if w.name == "longctx_tbq4":
        assert run.bulk == 512 * w.n_layers


def test_fullsize_records_rows_and_dequant(run):
    w = run.w
    for (layer, seq, h), (hc, refs, sealed, _) in run.oracle.items():
        where = f"layer {layer} seq {seq} head {h}"
        ng = (hc.S - 128) // 128
        for which, role in ((0, "K"), (1, "V")):
            body, off = _region(run.cache, layer, seq, h, which, _lib.REGION_BODY)
            _check_body(w, hc, body, role, ng, where)
            _check_journal(w, run.cache, hc, layer, seq, h, which, role, range(max(hc.S, 128), hc.N), where)
            _check_tail(w, run.cache, hc, layer, seq, h, which, role, where)
        _check_dequant(w, run.cache, hc, layer, seq, h, where)


def test_fullsize_offsets_beyond_2gib(run):
    """The last layer's sampled storage of the two large pools lies beyond 2 GiB of offset."""
    w = run.w
    if w.name not in ("fa14b_q8q4", "longctx_tbq4"):
        pytest.skip("pool under 2 GiB")
    seq, h = run.samples[0]
    ptr, _ = _lib.kv_region_ptr(run.cache.h, w.n_layers - 1, seq, h, 1, _lib.REGION_BODY)
    assert ptr - run.cache.pool.data_ptr() > (2 << 30)
    assert (w.n_layers - 1, seq, h) in run.oracle


def test_fullsize_attention_first_and_last_step(run):
    w = run.w
    G = w.G
    for (layer, seq, h), (hc, refs, sealed, _) in run.oracle.items():
        for s, got in ((0, run.first), (run.steps - 1, run.last)):
            tolerance.check(w.name, got[layer, seq, h * G:(h + 1) * G], refs[s],
                            where=f"step {s} layer {layer} seq {seq} head {h}")


def test_fullsize_prefill(run):
    """kv_prefill of the sampled sequences' whole contexts (the bench's prefill measurement)."""
    from quantized_kv_cache_gb300 import KVCache
    from quantized_kv_cache_gb300.runner import DeviceSynth
    w = run.w
    H, D = w.n_kv_heads, w.head_dim
    ds = DeviceSynth(w, 0)
    cache = KVCache(w.config(n_layers=1), 0)
    try:
        seqs = sorted({seq for seq, _ in run.samples})
        for seq in seqs:
            n0 = w.contexts[seq]
            k = torch.empty((1, n0, H, D), dtype=torch.float16, device=ds.dev)
            v = torch.empty_like(k)
            ds.kv(synth.T_K, 0, seq, 0, n0, k)
            ds.kv(synth.T_V, 0, seq, 0, n0, v)
            g = cache.prefill(0, [seq], k, v, w.keep)
            torch.cuda.synchronize()
            lim = n0 - w.keep - 128
            S1 = 128 + (lim // 128 * 128 if lim >= 128 else 0)
            assert cache.state(0, seq) == (n0, S1)
            assert g == (S1 - 128) // 128
            del k, v
        assert _lib.kv_get_status(cache.h) == 0
        for seq, h in run.samples:
            n0 = w.contexts[seq]
            S1 = cache.state(0, seq)[1]
            hc = copy.deepcopy(run.oracle[(0, seq, h)][3])   # the oracle right after the bench's prefill
            hc.seal(w.keep)
            assert (hc.N, hc.S) == (n0, S1)
            ng = (S1 - 128) // 128
            where = f"prefill seq {seq} head {h}"
            for which, role in ((0, "K"), (1, "V")):
                body, _ = _region(cache, 0, seq, h, which, _lib.REGION_BODY)
                _check_body(w, hc, body, role, ng, where)
                _check_journal(w, cache, hc, 0, seq, h, which, role, range(max(S1, 128, n0 - 4), n0), where)
                if w.journal == "tq6_0":
                    tail = _region(cache, 0, seq, h, which, _lib.REGION_TAIL)[0].view(np.uint16).reshape(w.tail, D)
                    pos = np.arange(max(S1, 128, n0 - 4), n0) % w.tail
                    assert np.array_equal(tail[pos], hc.tail[role][pos]), where
    finally:
        cache.close()
