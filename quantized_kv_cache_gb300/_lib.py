"""ctypes binding of libkvq.so — argument marshalling only.

Every function here forwards to the C ABI of the same name (include/kvq.h) and turns a
non-OK status into ``KVQError``. There is no fallback: if the shared library is missing
the import of a call raises, on every machine.
"""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libkvq.so")

# kvq_fmt
(F16, BF16, TQ6_0, TBQ4, Q8_0, Q4_0, KVARN4, KVARN5, KVARN2, KVARN3, KVARN6, KVARN8, Q5_0, Q6_0, Q4_1, Q5_1,
 TURBO3, TQ5_0) = range(18)
FMT_NAMES = {"f16": F16, "bf16": BF16, "tq6_0": TQ6_0, "tbq4": TBQ4, "q8_0": Q8_0, "q4_0": Q4_0,
             "kvarn4": KVARN4, "kvarn5": KVARN5, "kvarn2": KVARN2, "kvarn3": KVARN3, "kvarn6": KVARN6,
             "kvarn8": KVARN8, "q5_0": Q5_0, "q6_0": Q6_0, "q4_1": Q4_1, "q5_1": Q5_1, "turbo3": TURBO3,
             "tq5_0": TQ5_0}
# KVarN balancing rules (kvq_config.kvarn_balance)
KVARN_BALANCE = {"final16": 0, "best8": 1}
# regions
REGION_SINK, REGION_JOURNAL, REGION_JOURNAL_SCALE, REGION_TAIL, REGION_BODY = range(5)
ENOSPC = 2
STATUS = {0: "KVQ_OK", 1: "KVQ_EINVAL", 2: "KVQ_ENOSPC", 3: "KVQ_EUNSUPPORTED", 4: "KVQ_ECUDA", 5: "KVQ_EDEVICE"}


class KVQError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")


class kvq_config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("max_seqs", ctypes.c_int32), ("kvarn_balance", ctypes.c_int32),
                ("max_ctx", ctypes.c_int64), ("k_body", ctypes.c_int32), ("v_body", ctypes.c_int32),
                ("journal", ctypes.c_int32), ("tail_fmt", ctypes.c_int32), ("tail", ctypes.c_int32),
                ("ring_capacity", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
                ("reserved1", ctypes.c_int32)]


class kvq_bytes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("body_bytes_per_token", "f16_bytes_per_token",
                                               "journal_bytes_per_slot", "tail_bytes_per_slot", "sink_bytes",
                                               "fixed_bytes_per_seq", "pool_bytes")]


_lib = None

P = ctypes.c_void_p
I32 = ctypes.c_int32
I64 = ctypes.c_int64
SZ = ctypes.c_size_t

_SIGS = {
    "kv_bytes_per_token": [ctypes.POINTER(kvq_config), ctypes.POINTER(kvq_bytes)],
    "kv_required_bytes": [ctypes.POINTER(kvq_config), ctypes.POINTER(SZ), ctypes.POINTER(SZ)],
    "kv_auto_tier": [ctypes.POINTER(kvq_config), I64, ctypes.c_uint64, ctypes.POINTER(I32), ctypes.POINTER(I32),
                     ctypes.POINTER(ctypes.c_uint64)],
    "kv_tier_budget": [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.POINTER(ctypes.c_uint64)],
    "kv_create": [ctypes.POINTER(kvq_config), P, SZ, ctypes.c_int, ctypes.POINTER(P)],
    "kv_destroy": [P],
    "kv_reset": [P, ctypes.c_int, ctypes.c_int],
    "kv_append": [P, ctypes.c_int, ctypes.POINTER(I32), ctypes.c_int, ctypes.c_int, P, P, P],
    "kv_seal": [P, ctypes.c_int, ctypes.POINTER(I32), ctypes.c_int, ctypes.c_int, ctypes.POINTER(I64), P],
    "kv_prefill": [P, ctypes.c_int, ctypes.POINTER(I32), ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int,
                   ctypes.POINTER(I64), P],
    "kv_decode_attn": [P, ctypes.c_int, ctypes.POINTER(I32), ctypes.c_int, P, P, P, SZ, P],
    "kv_state": [P, ctypes.c_int, ctypes.c_int, ctypes.POINTER(I64), ctypes.POINTER(I64)],
    "kv_get_status": [P, ctypes.POINTER(ctypes.c_uint32)],
    "kv_dequant": [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, I64, I64, P, P],
    "kv_region_ptr": [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                      ctypes.POINTER(P), ctypes.POINTER(SZ)],
    "kv_format_tables": [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float),
                         ctypes.POINTER(ctypes.c_uint64)],
    "kv_format_tables_turbo3": [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)],
    "kv_prefill_plan": [I64, I64, I64, ctypes.c_int32, ctypes.c_int32, I64, ctypes.POINTER(I64)],
    "kv_decode_step": [P, ctypes.c_int, ctypes.POINTER(I32), ctypes.c_int, P, P, P, P, ctypes.c_int, ctypes.c_int,
                       P, SZ, ctypes.POINTER(P), ctypes.POINTER(I64), P],
    "kv_decode_attn_noalloc": [P, ctypes.c_int, ctypes.POINTER(I32), ctypes.c_int, P, P, P],
    "kv_set_graph_mode": [P, ctypes.c_int],
    "kv_snapshot_size": [P, ctypes.POINTER(SZ)],
    "kv_snapshot": [P, P, SZ],
    "kv_restore": [P, P, SZ],
    "kv_test_wait_timeout": [P, ctypes.c_uint64, P],
    "kvq_synth_fill": [P, I64, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_uint64), I64, P, P, P],
}


def load(path=LIB_PATH):
    """Load libkvq.so (built by ``quantized_kv_cache_gb300.build``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libkvq.so not found at {path}: build it with quantized_kv_cache_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, args in _SIGS.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.kv_status_string.argtypes = [ctypes.c_int]
    lib.kv_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def exported_symbols():
    return list(_SIGS) + ["kv_status_string"]


def _check(name, code):
    if code != 0:
        raise KVQError(name, code)


def _ids(seq_ids):
    arr = (I32 * len(seq_ids))(*[int(s) for s in seq_ids])
    return arr, len(seq_ids)


def kv_bytes_per_token(cfg):
    out = kvq_bytes()
    _check("kv_bytes_per_token", load().kv_bytes_per_token(ctypes.byref(cfg), ctypes.byref(out)))
    return {f: getattr(out, f) for f, _ in kvq_bytes._fields_}


def kv_auto_tier(cfg, tokens, budget_bytes):
    """(k_fmt, v_fmt, cost_bytes, fits): the ladder rung kv_auto_tier picks."""
    k, v, cost = I32(), I32(), ctypes.c_uint64()
    code = load().kv_auto_tier(ctypes.byref(cfg), tokens, budget_bytes, ctypes.byref(k), ctypes.byref(v),
                               ctypes.byref(cost))
    if code not in (0, ENOSPC):
        raise KVQError("kv_auto_tier", code)
    return k.value, v.value, cost.value, code == 0


def kv_tier_budget(free_bytes, resident_bytes, target_bytes=0):
    out = ctypes.c_uint64()
    _check("kv_tier_budget", load().kv_tier_budget(free_bytes, resident_bytes, target_bytes, ctypes.byref(out)))
    return out.value


def kv_required_bytes(cfg):
    pool, ws = SZ(), SZ()
    _check("kv_required_bytes", load().kv_required_bytes(ctypes.byref(cfg), ctypes.byref(pool), ctypes.byref(ws)))
    return pool.value, ws.value


def kv_create(cfg, pool_ptr, pool_bytes, device):
    h = P()
    _check("kv_create", load().kv_create(ctypes.byref(cfg), P(pool_ptr), pool_bytes, device, ctypes.byref(h)))
    return h


def kv_destroy(h):
    _check("kv_destroy", load().kv_destroy(h))


def kv_reset(h, layer, seq):
    _check("kv_reset", load().kv_reset(h, layer, seq))


def kv_append(h, layer, seq_ids, n_tok, k_ptr, v_ptr, stream=0):
    ids, n = _ids(seq_ids)
    _check("kv_append", load().kv_append(h, layer, ids, n, n_tok, P(k_ptr), P(v_ptr), P(stream)))


def kv_prefill(h, layer, seq_ids, n_tok, k_ptr, v_ptr, keep, stream=0):
    ids, n = _ids(seq_ids)
    g = I64()
    _check("kv_prefill", load().kv_prefill(h, layer, ids, n, n_tok, P(k_ptr), P(v_ptr), keep, ctypes.byref(g),
                                           P(stream)))
    return g.value


def kv_seal(h, layer, seq_ids, keep, stream=0):
    ids, n = _ids(seq_ids)
    g = I64()
    _check("kv_seal", load().kv_seal(h, layer, ids, n, keep, ctypes.byref(g), P(stream)))
    return g.value


def kv_decode_attn(h, layer, seq_ids, q_ptr, out_ptr, ws_ptr, ws_bytes, stream=0):
    ids, n = _ids(seq_ids)
    _check("kv_decode_attn", load().kv_decode_attn(h, layer, ids, n, P(q_ptr), P(out_ptr), P(ws_ptr), ws_bytes,
                                                   P(stream)))


def kv_decode_step(h, n_layers, seq_ids, q_ptr, k_ptr, v_ptr, out_ptr, seal_trigger, keep, ws_ptr, ws_bytes,
                   events=None, stream=0):
    """events: None or a list of 2 * n_layers raw cudaEvent_t handles (ints)."""
    ids, n = _ids(seq_ids)
    ev = None
    if events is not None:
        ev = (P * len(events))(*[P(e) for e in events])
    g = I64()
    _check("kv_decode_step", load().kv_decode_step(h, n_layers, ids, n, P(q_ptr), P(k_ptr), P(v_ptr), P(out_ptr),
                                                   seal_trigger, keep, P(ws_ptr), ws_bytes, ev, ctypes.byref(g),
                                                   P(stream)))
    return g.value


def kv_set_graph_mode(h, enable):
    """Whether kv_decode_step replays its launches as one CUDA graph (default on)."""
    _check("kv_set_graph_mode", load().kv_set_graph_mode(h, 1 if enable else 0))


def kv_decode_attn_noalloc(h, layer, seq_ids, q_ptr, out_ptr, stream=0):
    """kv_decode_attn without a caller workspace (the library's fixed device array)."""
    ids, n = _ids(seq_ids)
    _check("kv_decode_attn_noalloc", load().kv_decode_attn_noalloc(h, layer, ids, n, P(q_ptr), P(out_ptr),
                                                                   P(stream)))


def kv_snapshot(h):
    n = SZ()
    _check("kv_snapshot_size", load().kv_snapshot_size(h, ctypes.byref(n)))
    buf = ctypes.create_string_buffer(n.value)
    _check("kv_snapshot", load().kv_snapshot(h, buf, n.value))
    return buf


def kv_restore(h, buf):
    _check("kv_restore", load().kv_restore(h, buf, len(buf)))


def kv_state(h, layer, seq):
    n, s = I64(), I64()
    _check("kv_state", load().kv_state(h, layer, seq, ctypes.byref(n), ctypes.byref(s)))
    return n.value, s.value


def kv_get_status(h):
    w = ctypes.c_uint32()
    code = load().kv_get_status(h, ctypes.byref(w))
    if code not in (0, 5):
        raise KVQError("kv_get_status", code)
    return w.value


def kv_test_wait_timeout(h, limit_ns, stream=0):
    _check("kv_test_wait_timeout", load().kv_test_wait_timeout(h, limit_ns, P(stream)))


def kv_dequant(h, layer, seq, head, which, p0, n, out_ptr, stream=0):
    _check("kv_dequant", load().kv_dequant(h, layer, seq, head, which, p0, n, P(out_ptr), P(stream)))


def kv_region_ptr(h, layer, seq, head, which, region):
    ptr, nb = P(), SZ()
    _check("kv_region_ptr", load().kv_region_ptr(h, layer, seq, head, which, region, ctypes.byref(ptr),
                                                 ctypes.byref(nb)))
    return ptr.value, nb.value


def kv_format_tables():
    c = (ctypes.c_float * 16)()
    b = (ctypes.c_float * 15)()
    s = (ctypes.c_uint64 * 4)()
    _check("kv_format_tables", load().kv_format_tables(c, b, s))
    return list(c), list(b), list(s)


def kv_prefill_plan(n_tokens, sealed_end, n_tok, keep, ring_capacity, max_ctx):
    """The 8 range bounds of kv_prefill's plan (head, journal seal, direct seal, rest)."""
    r = (I64 * 8)()
    _check("kv_prefill_plan", load().kv_prefill_plan(n_tokens, sealed_end, n_tok, keep, ring_capacity, max_ctx, r))
    return list(r)


def kv_format_tables_turbo3():
    c = (ctypes.c_float * 8)()
    b = (ctypes.c_float * 7)()
    _check("kv_format_tables_turbo3", load().kv_format_tables_turbo3(c, b))
    return list(c), list(b)


def kvq_synth_fill(out_ptr, n_pos, n_heads, head_dim, head_keys, pos0, factor_ptr, table_ptr, stream=0):
    keys = (ctypes.c_uint64 * len(head_keys))(*[int(k) for k in head_keys])
    _check("kvq_synth_fill", load().kvq_synth_fill(P(out_ptr), n_pos, n_heads, head_dim, keys, pos0,
                                                   P(factor_ptr or 0), P(table_ptr), P(stream)))
