"""GPU parity at the workloads' full sizes, in the launch configuration the bench times.

For each workload (one layer of it: the kernels run per layer, so one layer has every other
dimension at full size), the GPU cache is built the way ``bench.py`` builds it: the
device-side seeded generator fills the rows, the bench's prefill plan appends and seals them,
and one decode step runs through ``kv_decode_step`` (the CUDA-graph path: append, seal per
policy, decode attention and merge). For sampled (sequence, KV head) pairs the oracle replays
the same appends and seals from the host-side generator (the same counter-based streams) and
the test compares:

- the sequence's lengths (N, S);
- every body record of the sampled heads (K and V) byte for byte;
- the newest journal rows (tq6_0 codes and scales, or exact rows) and exact-tail rows;
- the decode output of the head's query group against the fp64 oracle attention over the
  same regions, within the decode tolerance |gpu - oracle| <= 1e-3 + 2e-3 |oracle|;
- the bench's prefill measurement: kv_prefill of a sampled sequence's whole context into a fresh
  one-layer cache; lengths, the sealed records (a record depends only on its group's rows, so
  the oracle's cache above, sealed on, holds the same ones) and the newest journal and tail rows.
"""

import copy
import dataclasses

import numpy as np
import pytest

from oracle import attention
from oracle.cache import HeadCache, HeadConfig
from quantized_kv_cache_gb300 import configs, synth, _lib

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-3, 2e-3

# workload -> sampled (sequence, KV head) pairs
SAMPLES = {
    "tiny_tbq4": [(0, 0), (0, 1)],
    "hybrid27b_kvarn44": [(0, 3)],
    "fa14b_q8q4": [(0, 5)],
    "widehead_kvarn55": [(2, 1), (7, 0)],
    "longctx_tbq4": [(0, 2), (3, 0)],
    "hybrid27b_kvarn32_200k": [(0, 2)],
    "fa14b_q51q40": [(0, 3)],
    "hybrid27b_tq50tbq4_110k": [(0, 1)],
}


def _step_trigger(w):
    """Seal trigger of the decode step: tiny_tbq4's recipe seals its 6 groups in the step
    (after the append, before the attention); the other workloads follow their policy."""
    return 0 if w.seal_trigger == -1 else w.seal_trigger


def _gpu_run(w):
    from quantized_kv_cache_gb300 import KVCache
    from quantized_kv_cache_gb300.runner import DeviceSynth, DecodeInputs, build_state
    dev = torch.device("cuda", 0)
    cfg = w.config()
    cfg.max_ctx = max(w.contexts) + 1 + 512
    cache = KVCache(cfg, 0)
    ds = DeviceSynth(w, 0)
    seq_ids = list(range(len(w.contexts)))
    stream = torch.cuda.current_stream(dev).cuda_stream
    build_state(w, cache, ds, seq_ids, [0], stream=stream)
    inp = DecodeInputs(w, ds, seq_ids, w.contexts, 1, [0])
    out = torch.empty((1, len(seq_ids), w.n_q_heads, w.head_dim), dtype=torch.float16, device=dev)
    _lib.kv_decode_step(cache.h, 1, seq_ids, inp.q[0].data_ptr(), inp.k[0].data_ptr(), inp.v[0].data_ptr(),
                        out.data_ptr(), _step_trigger(w), w.keep, cache.ws.data_ptr(), cache.ws_bytes, None, stream)
    torch.cuda.synchronize()
    st = _lib.kv_get_status(cache.h)
    return cache, inp, out.cpu().numpy()[0], st


_HEADS = {}


def _oracle_head(w, seq, h):
    """The oracle's cache of (layer 0, seq, h) after the bench's prefill and one decode step."""
    key = (w.name, seq, h)
    if key not in _HEADS:
        _HEADS[key] = _replay(w, seq, h)
    return _HEADS[key]


def _replay(w, seq, h):
    from quantized_kv_cache_gb300.runner import prefill_plan
    D = w.head_dim
    hc = HeadCache(HeadConfig(D, w.k_body, w.v_body, w.journal, w.tail_fmt, w.tail, w.ring))
    n0 = w.contexts[seq]

    def rows(p0, n):
        k = synth.kv_values(w.seed, synth.T_K, 0, seq, h, p0, n, D, w.n_out, w.out_factor)
        v = synth.kv_values(w.seed, synth.T_V, 0, seq, h, p0, n, D)
        return k, v

    pos = 0
    for c, seal in prefill_plan(w, n0):
        hc.append(*rows(pos, c))
        pos += c
        if seal:
            hc.seal(w.keep)
    hc.append(*rows(n0, 1))
    if configs.should_seal(dataclasses.replace(w, seal_trigger=_step_trigger(w)), hc.N, hc.S):
        hc.seal(w.keep)
    return hc


def _check_records(w, hc, body, role, groups, where):
    rb = len(hc.record_bytes(0, role))
    for g in groups:
        got = body[g * rb:(g + 1) * rb]
        diff = np.flatnonzero(got != hc.record_bytes(g, role))
        assert diff.size == 0, f"{w.name} {where} {role} group {g}: {diff.size} bytes differ, first {diff[:6]}"


def _region_bytes(cache, seq, head, which, region):
    ptr, nb = _lib.kv_region_ptr(cache.h, 0, seq, head, which, region)
    off = ptr - cache.pool.data_ptr()
    assert 0 <= off and off + nb <= cache.pool_bytes
    return cache.pool[off:off + nb].cpu().numpy()


@pytest.fixture(scope="module", params=list(SAMPLES))
def run(request):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = dataclasses.replace(configs.WORKLOADS[request.param], n_layers=1)
    cache, inp, out, status = _gpu_run(w)
    yield w, cache, inp, out, status
    cache.close()


def test_fullsize_inputs_and_status(run):
    w, cache, inp, out, status = run
    assert status == 0
    # the device generator draws the host generator's values (the oracle's inputs)
    for seq in range(len(w.contexts)):
        q = synth.q_values(w.seed, 0, seq, 0, w.n_q_heads, w.head_dim)
        assert np.array_equal(inp.q[0, 0, seq].cpu().numpy().view(np.uint16), q.view(np.uint16))
    assert np.all(np.isfinite(out))


def test_fullsize_sampled_records_and_rows(run):
    w, cache, inp, out, status = run
    D = w.head_dim
    for seq, h in SAMPLES[w.name]:
        hc = _oracle_head(w, seq, h)
        assert cache.state(0, seq) == (hc.N, hc.S), (seq, h)
        ng = (hc.S - 128) // 128
        for wi, role in ((0, "K"), (1, "V")):
            if ng:
                body = _region_bytes(cache, seq, h, wi, _lib.REGION_BODY)
                _check_records(w, hc, body, role, range(ng), f"seq {seq} head {h}")
            # the newest positions of the journal (and the exact tail with a tq6_0 ring)
            newest = range(max(hc.S, hc.N - 4), hc.N)
            if w.journal == "tq6_0":
                codes = _region_bytes(cache, seq, h, wi, _lib.REGION_JOURNAL).reshape(w.ring, D // 128, 96)
                sc = _region_bytes(cache, seq, h, wi, _lib.REGION_JOURNAL_SCALE).view(np.uint16).reshape(w.ring, D // 128)
                tail = _region_bytes(cache, seq, h, wi, _lib.REGION_TAIL).view(np.uint16).reshape(w.tail, D)
                for p in newest:
                    d, ql, qh = hc.tq6_slot_bytes(p, role)
                    slot = (p - 128) % w.ring
                    assert np.array_equal(codes[slot], np.concatenate([ql, qh], axis=1)), (seq, h, role, p)
                    assert np.array_equal(sc[slot], d.view(np.uint16)), (seq, h, role, p)
                    assert np.array_equal(tail[p % w.tail], hc.tail[role][p % w.tail]), (seq, h, role, p)
            else:
                jx = _region_bytes(cache, seq, h, wi, _lib.REGION_JOURNAL).view(np.uint16).reshape(w.ring, D)
                for p in newest:
                    slot = (p - 128) % w.ring
                    assert np.array_equal(jx[slot], hc.jx[role][slot]), (seq, h, role, p)


def test_fullsize_sampled_attention(run):
    w, cache, inp, out, status = run
    G = w.n_q_heads // w.n_kv_heads
    D = w.head_dim
    for seq, h in SAMPLES[w.name]:
        hc = _oracle_head(w, seq, h)
        q = synth.q_values(w.seed, 0, seq, 0, w.n_q_heads, D)[h * G:(h + 1) * G].astype(np.float64)
        ref = attention.attend(q, hc.regions(), hc.cfg.rot, 1.0 / np.sqrt(D))
        got = out[seq, h * G:(h + 1) * G].astype(np.float64)
        err = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
        assert np.all(err <= 0), f"{w.name} seq {seq} head {h}: excess {err.max():.3g}"


def test_fullsize_bulk_seal(run):
    """The bulk seal of longctx_tbq4 (every sequence's groups older than the newest keep, one
    launch): the sampled heads' new records against the oracle's seal of the same groups."""
    w, cache, inp, out, status = run
    if w.name != "longctx_tbq4":
        pytest.skip("the bulk seal belongs to longctx_tbq4")
    seq_ids = list(range(len(w.contexts)))
    before = {seq: cache.state(0, seq)[1] for seq in seq_ids}
    groups = _lib.kv_seal(cache.h, -1, seq_ids, w.keep, 0)
    torch.cuda.synchronize()
    assert _lib.kv_get_status(cache.h) == 0
    assert groups == sum((cache.state(0, s)[1] - before[s]) // 128 for s in seq_ids) == 512
    for seq, h in SAMPLES[w.name]:
        hc = _oracle_head(w, seq, h)
        g0 = (hc.S - 128) // 128
        hc.seal(w.keep)
        assert cache.state(0, seq) == (hc.N, hc.S)
        g1 = (hc.S - 128) // 128
        for wi, role in ((0, "K"), (1, "V")):
            body = _region_bytes(cache, seq, h, wi, _lib.REGION_BODY)
            _check_records(w, hc, body, role, range(g0, g1), f"bulk seal seq {seq} head {h}")


def test_fullsize_prefill(run):
    """kv_prefill of the sampled sequences' whole contexts (the bench's prefill measurement)."""
    from quantized_kv_cache_gb300 import KVCache
    from quantized_kv_cache_gb300.runner import DeviceSynth
    w = run[0]
    H, D = w.n_kv_heads, w.head_dim
    ds = DeviceSynth(w, 0)
    cache = KVCache(w.config(n_layers=1), 0)
    try:
        seqs = sorted({seq for seq, _ in SAMPLES[w.name]})
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
        for seq, h in SAMPLES[w.name]:
            n0 = w.contexts[seq]
            S1 = cache.state(0, seq)[1]
            hc = copy.deepcopy(_oracle_head(w, seq, h))   # n0 + 1 positions
            if hc.S < S1:
                hc.seal(w.keep)
            assert hc.S >= S1
            ng = (S1 - 128) // 128
            for wi, role in ((0, "K"), (1, "V")):
                if ng:
                    body = _region_bytes(cache, seq, h, wi, _lib.REGION_BODY)
                    _check_records(w, hc, body, role, sorted({0, ng // 2, ng - 1}) if ng > 3 else range(ng),
                                   f"prefill seq {seq} head {h}")
                    if ng > 3:   # every record, cheaply: the whole sealed body in one comparison
                        rb = len(hc.record_bytes(0, role))
                        ref = np.concatenate([hc.record_bytes(gg, role) for gg in range(ng)])
                        assert np.array_equal(body[:ng * rb], ref), f"prefill seq {seq} head {h} {role} body"
                newest = range(max(S1, n0 - 4), n0)
                if w.journal == "tq6_0":
                    codes = _region_bytes(cache, seq, h, wi, _lib.REGION_JOURNAL).reshape(w.ring, D // 128, 96)
                    sc = _region_bytes(cache, seq, h, wi, _lib.REGION_JOURNAL_SCALE).view(np.uint16).reshape(w.ring, D // 128)
                    tail = _region_bytes(cache, seq, h, wi, _lib.REGION_TAIL).view(np.uint16).reshape(w.tail, D)
                    for p in newest:
                        d, ql, qh = hc.tq6_slot_bytes(p, role)
                        slot = (p - 128) % w.ring
                        assert np.array_equal(codes[slot], np.concatenate([ql, qh], axis=1)), (seq, h, role, p)
                        assert np.array_equal(sc[slot], d.view(np.uint16)), (seq, h, role, p)
                        assert np.array_equal(tail[p % w.tail], hc.tail[role][p % w.tail]), (seq, h, role, p)
                else:
                    jx = _region_bytes(cache, seq, h, wi, _lib.REGION_JOURNAL).view(np.uint16).reshape(w.ring, D)
                    for p in newest:
                        slot = (p - 128) % w.ring
                        assert np.array_equal(jx[slot], hc.jx[role][slot]), (seq, h, role, p)
    finally:
        cache.close()
