#!/usr/bin/env python3
"""Benchmark of the rotated low-bit KV cache hot path on GB300.

One step = one decode step over every layer of the workload: append one position per
sequence (rotate + tq6_0 staging or exact copy), seal when the seal policy asks, and
decode attention over every region (split-K + log-sum-exp merge). The metric is the
decode attention's effective KV bandwidth: the bytes the method must read (sink, body
records, tq6_0 ring span, exact tail, q and out) divided by the time of the whole step.

Default workload (the headline): longctx_tbq4 (4 sequences at 262,144 / 196,608 / 131,072 /
65,536 positions, 16 layers, 4 KV heads x 256, 24 query heads, TBQ4 body, tq6_0 ring,
1,024-position exact tail; its bulk seal of 512 groups per layer timed alone, and the decode
after it). The same line carries blocks for fa14b_q8q4 (48 layers, 8 KV heads x 128, 131,072
positions, Q8_0 K / Q4_0 V) and hybrid27b_kvarn44 (16 layers, 4 KV heads x 256, 32,768
positions, KVarN 4/4), each with its decode, roofline and seal figures. Prints one JSON line
(rank 0).

--impl reference times the CPU oracle (numpy, fp64 attention) on a bounded sample of the
same workload, spread over the host's cores: the reference the CUDA path is checked against.
"""

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn effective KV GB/s (% of GB300 HBM peak); seal groups/s; 32k-262k ctx"
UNIT = "GB/s"
DEFAULT_WORKLOAD = "longctx_tbq4"
# further workloads measured in the same run when the headline is the default one
EXTRA_WORKLOADS = ("fa14b_q8q4", "hybrid27b_kvarn44")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed decode steps (default: the workload's own count)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="measure the headline workload only")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first N layers (a smaller case for profiling; the line names it)")
    args = ap.parse_args()
    if args.steps <= 0 and args.workload in _workloads():
        args.steps = _workloads()[args.workload].steps
    return args


def _workloads():
    from quantized_kv_cache_gb300 import configs
    return configs.WORKLOADS


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# DRAM bytes (read + write) per launch of decode_attn_kernel, from one ncu launch-list capture
# per workload at the same per-layer shape (--layers 1 or 2), with the hash of the decode
# kernel's sources they were taken from: once those sources change, the figure is stale and
# the line reports null until a new capture replaces it.
DECODE_SOURCES = ("kernels_body.cu", "region_item.cuh", "stream_common.cuh", "device_common.cuh", "append_row.cuh")
MEASURED_TRAFFIC = {
    "hybrid27b_kvarn44": (42.88e6, "e4787c2cf91b"),
    "fa14b_q8q4": (222.05e6, "e4787c2cf91b"),
    "longctx_tbq4": (750.91e6, "e4787c2cf91b"),
    "widehead_kvarn55": (193.74e6, "e4787c2cf91b"),
    "hybrid27b_kvarn32_200k": (156.86e6, "e4787c2cf91b"),
    "fa14b_q51q40": (180.38e6, "e4787c2cf91b"),
    "hybrid27b_tq50tbq4_110k": (140.15e6, "e4787c2cf91b"),
}


def decode_sources_sha():
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        with open(os.path.join(ROOT, "quantized_kv_cache_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def measured_traffic(name):
    t = MEASURED_TRAFFIC.get(name)
    if t is None or t[1] != decode_sources_sha():
        return None
    return t[0]


# --------------------------------------------------------------------------- byte model
def layer_step_bytes(w, states):
    """Algorithmic bytes one decode attention of one layer reads and writes.

    states: list of (N, S) per sequence after the step's append and seal. Per KV head:
    sink positions x 2 D x 2 B, body positions x (K + V record bytes) / 128, tq6_0 ring
    span x 2 x (D/128) x 98 B, exact tail (or exact journal) positions x 2 D x 2 B; plus the
    fp16 query and output of every sequence.
    """
    from quantized_kv_cache_gb300.configs import record_bytes
    D, H = w.head_dim, w.n_kv_heads
    rec = record_bytes(w.k_body, D) + record_bytes(w.v_body, D)
    total = 0
    for N, S in states:
        sink = min(N, 128)
        body = max(S - 128, 0)
        if w.journal == "tq6_0":
            E = max(S, N - w.tail)
            ring, exact = E - S, N - max(E, 128)
            per_head = sink * 4 * D + body * rec // 128 + ring * 2 * (D // 128) * 98 + exact * 4 * D
        else:
            exact = N - max(S, 128)
            per_head = sink * 4 * D + body * rec // 128 + exact * 4 * D
        total += H * per_head + 2 * w.n_q_heads * D * 2
    return total


def initial_states(w, contexts):
    """(N, S) per sequence after prefill (the workload's starting state)."""
    from quantized_kv_cache_gb300.configs import groups_to_seal
    from quantized_kv_cache_gb300.runner import prefill_plan
    cur = []
    for n0 in contexts:
        n, S = 0, 128
        for c, seal in prefill_plan(w, n0):
            n += c
            if seal:
                S += 128 * groups_to_seal(n, S, w.keep)
        cur.append((n, S))
    return cur


def simulate_states(w, contexts, steps):
    """(N, S) per sequence after each step's append and seal, following the seal policy."""
    from quantized_kv_cache_gb300.configs import should_seal, groups_to_seal
    cur = [list(s) for s in initial_states(w, contexts)]
    out = []
    for _ in range(steps):
        for st in cur:
            st[0] += 1
            if should_seal(w, st[0], st[1]):
                st[1] += 128 * groups_to_seal(st[0], st[1], w.keep)
        out.append([tuple(s) for s in cur])
    return out


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.device = device
        self.samples = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.device), "--query-gpu=timestamp," + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if t0 - 0.02 <= r[0] <= t1 + 0.02]
        use = inside or rows[-5:]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        sm = [float(p[1]) for _, p in use if p[1].replace(".", "").isdigit()]
        mx = [float(p[2]) for _, p in use if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, p in use:
            for n, v in zip(names, p[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(use), "in_timed_window": bool(inside)}


# --------------------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import __graft_entry__
    __graft_entry__.build()

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    result = measure_workload(args.workload, args, world, local_rank, clocks, headline=True)
    if not args.no_extra and args.workload == DEFAULT_WORKLOAD and not args.layers:
        result["workloads"] = {name: measure_workload(name, args, world, local_rank, clocks, headline=False)
                               for name in EXTRA_WORKLOADS}
    clocks.stop()
    result["clocks"] = clocks.summary(*result.pop("_window"))
    for blk in result.get("workloads", {}).values():
        blk["clocks"] = clocks.summary(*blk.pop("_window"))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.workload, steps=4)
    return result


def measure_workload(name, args, world, local_rank, clocks, headline):
    """Builds one workload's cache on the device, times K decode steps (the headline pass),
    then the same steps with events around every decode kernel (the roofline), the seal, the
    prefill and (headline only) the end-to-end pass with host buffers. Frees the cache."""
    import torch
    import quantized_kv_cache_gb300 as pkg
    from quantized_kv_cache_gb300 import configs, _lib
    from quantized_kv_cache_gb300.runner import DeviceSynth, DecodeInputs, build_state

    dev = torch.device("cuda", local_rank)
    w = configs.WORKLOADS[name]
    if args.layers:
        w = dataclasses.replace(w, n_layers=min(args.layers, w.n_layers))
    K, W = args.steps, args.warmup
    n_steps = max(K, W, w.steps)
    seq_ids = list(range(len(w.contexts)))
    cfg = w.config()
    cfg.max_ctx = max(w.contexts) + n_steps + 512 + 32 * 128   # room for the bulk-seal groups
    cache = pkg.KVCache(cfg, local_rank)
    ds = DeviceSynth(w, local_rank)
    layers = list(range(w.n_layers))
    stream = torch.cuda.current_stream(dev).cuda_stream
    build_state(w, cache, ds, seq_ids, layers, stream=stream)
    inp = DecodeInputs(w, ds, seq_ids, w.contexts, n_steps, layers)
    out = torch.empty((w.n_layers, len(seq_ids), w.n_q_heads, w.head_dim), dtype=torch.float16, device=dev)
    torch.cuda.synchronize()
    snap = _lib.kv_snapshot(cache.h)
    pool_backup = cache.pool.clone()

    def restore():
        torch.cuda.synchronize()
        _lib.kv_restore(cache.h, snap)
        cache.pool.copy_(pool_backup)
        torch.cuda.synchronize()

    def step(s, events=None):
        return _lib.kv_decode_step(cache.h, w.n_layers, seq_ids, inp.q[s].data_ptr(), inp.k[s].data_ptr(),
                                   inp.v[s].data_ptr(), out.data_ptr(), w.seal_trigger, w.keep,
                                   cache.ws.data_ptr(), cache.ws_bytes, events, stream)

    for s in range(W):
        step(s)
    restore()

    # events around every attention launch of the timed region (recorded by the library)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * w.n_layers)] for _ in range(K)]
    for row in evs:
        for e in row:
            e.record()
    torch.cuda.synchronize()
    handles = [[e.cuda_event for e in row] for row in evs]

    dist_barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    torch.cuda.nvtx.range_push("timed")
    t_start.record()
    sealed = 0
    for s in range(K):
        sealed += step(s)
    t_end.record()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    wall1 = time.time()
    dist_barrier(world)
    elapsed = t_start.elapsed_time(t_end) / 1e3
    elapsed_max = dist_max(elapsed, world)

    # the same K steps again from the same state, with events around every attention call
    # (recorded by the library inside the step): the per-call durations of the roofline. Kept
    # out of the headline pass, whose step is then one uninterrupted chain of launches.
    restore()
    torch.cuda.synchronize()
    for s in range(K):
        step(s, handles[s])
    torch.cuda.synchronize()

    states = simulate_states(w, w.contexts, K)
    step_bytes = [layer_step_bytes(w, st) for st in states]          # per layer-step, same for every layer
    total_bytes = sum(step_bytes) * w.n_layers
    attn_times = [evs[s][2 * l].elapsed_time(evs[s][2 * l + 1]) / 1e3 for s in range(K) for l in range(w.n_layers)]
    attn_bytes = [step_bytes[s] for s in range(K) for _ in range(w.n_layers)]
    hbm, peak_src = peaks()
    achieved = sum(attn_bytes) / sum(attn_times) / 1e9
    value = weak_value(total_bytes, elapsed_max, world)
    kernel_ms = 1e3 * sum(attn_times) / K

    seal = measure_seal(w, cache, inp, seq_ids, out, restore, stream, K, ds)
    prefill = measure_prefill(w, ds, seq_ids, stream)

    e2e = None
    if headline and not args.no_e2e:
        restore()
        e2e = measure_e2e(w, cache, inp, seq_ids, out, stream, K, total_bytes, world)

    launches = K * w.n_layers * launches_per_layer(w) + seal_launches(w, states)
    ms_step = elapsed_max / K * 1e3
    roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4),
                "traffic": measured_traffic(w.name),
                "kernel": "decode_attn_kernel: one layer's body and region items (and, in the decode "
                          "step, its append), timed by events recorded around its launch on the "
                          "calling stream in a second pass over the same K steps; bytes: the layer's "
                          "algorithmic bytes (KV regions, q, out)",
                "peak_source": f"{peak_src} hbm_gbs",
                "launches_timed": len(attn_times),
                "mean_launch_us": round(1e6 * sum(attn_times) / len(attn_times), 3),
                "algorithmic_bytes_per_launch": int(sum(attn_bytes) / len(attn_bytes)),
                "kernel_ms_per_step": round(kernel_ms, 4),
                "step_frac": round(value / world / hbm, 4)}
    res = {"value": round(value, 2), "unit": UNIT, "steps": K, "ms_per_step": round(ms_step, 4),
           "us_per_layer_step": round(1e3 * ms_step / w.n_layers, 3),
           "pct_of_hbm_peak": round(100 * value / world / hbm, 2),
           "config": config_block(w, K), "roofline": roofline, "seal": seal, "prefill": prefill,
           "groups_sealed_in_timed_region": sealed, "gpu_launches": launches, "_window": (wall0, wall1)}
    if e2e:
        res["e2e"] = e2e
    if headline:
        res = {"metric": METRIC, "value": res.pop("value"), "unit": UNIT, "n_gpus": world, "steps": K,
               "warmup": W, "ms_per_step": res.pop("ms_per_step"), "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "f16", "data": "synthetic", **res}
    cache.close()
    del cache, inp, out, pool_backup
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


# (head_dim, query tile, K body, V body) of the streaming decode kernel's instances
# (kernels_body.cu, the dispatch table); other layouts take the generic path
STREAMING = {(128, 8, "tbq4", "tbq4"), (256, 8, "tbq4", "tbq4"), (256, 16, "tbq4", "tbq4"),
             (128, 8, "q8_0", "q4_0"), (128, 16, "q8_0", "q4_0"), (256, 8, "kvarn4", "kvarn4"),
             (256, 16, "kvarn4", "kvarn4"), (512, 8, "kvarn5", "kvarn5"), (512, 16, "kvarn5", "kvarn5"),
             (256, 8, "kvarn3", "kvarn2"), (128, 8, "q5_1", "q4_0"), (256, 8, "tq5_0", "tbq4")}


def launches_per_layer(w):
    """Kernel launches of one layer's decode step outside seals: the decode kernel (which also
    appends the step's position) and the merge; on the generic path an append, the generic
    decode kernel and the merge."""
    nq = 8 if w.G <= 8 else 16
    fused = (w.head_dim, nq, w.k_body, w.v_body) in STREAMING and not (w.head_dim == 512 and w.journal == "tq6_0")
    return 2 if fused else 3


def seal_launches(w, states):
    """Seal launches of the steps: where the decode kernel appends (every layer in lockstep), a
    step's seals are one call over all layers, one launch; otherwise one launch per layer."""
    n = 0
    prev = None
    for st in states:
        if prev is not None:
            for (a, s0), (b, s1) in zip(prev, st):
                if s1 != s0:
                    n += 1 if launches_per_layer(w) == 2 else w.n_layers
                    break
        prev = st
    return n


# fp32 operations of the KVarN seal per encoded value: 16 balancing passes x (sum, deviation,
# square, variance sum, scale) + rounding (divide by C, subtract Z, scale by 1/S, rint, and the
# row min / max); plus the tq6_0 dequantize (1) or the HAD256 rotation of a 16-bit row (8 + 1)
KVARN_OPS_PER_VALUE = 16 * 5 + 6
KVARN_TQ6_OPS = 1
KVARN_ROT_OPS = 9
FP32_PEAK_TOPS = round(152 * 128 * 2.070e9 / 1e12, 2)


def bulk_seal_prefill(w, cache, ds, seq_ids, stream, max_groups=32):
    """Appends, to every sequence of every layer, as many whole groups (at most max_groups)
    as its journal has room for beyond the newest keep positions. Returns the groups added."""
    import torch
    from quantized_kv_cache_gb300 import synth
    H, D = w.n_kv_heads, w.head_dim
    added = 0
    buf_k = buf_v = None
    for layer in range(w.n_layers):
        for seq in seq_ids:
            N, S = cache.state(layer, seq)
            room = w.ring - (max(N, 128) - S)
            g = max(0, min(max_groups, room // 128))
            n = 128 * g
            if n == 0:
                continue
            if buf_k is None or buf_k.numel() < n * H * D:
                buf_k = torch.empty(n * H * D, dtype=torch.float16, device=ds.dev)
                buf_v = torch.empty_like(buf_k)
            ds.kv(synth.T_K, layer, seq, N, n, buf_k, stream)
            ds.kv(synth.T_V, layer, seq, N, n, buf_v, stream)
            cache.append(layer, [seq], buf_k[:n * H * D].view(1, n, H, D), buf_v[:n * H * D].view(1, n, H, D), stream)
            added += g
    return added


def measure_seal(w, cache, inp, seq_ids, out, restore, stream, K, ds=None):
    """Seal groups/s: time kv_seal calls alone with CUDA events."""
    import torch
    from quantized_kv_cache_gb300 import _lib
    from quantized_kv_cache_gb300.configs import should_seal, groups_to_seal
    restore()
    states = [initial_states(w, w.contexts)] + simulate_states(w, w.contexts, max(K, w.steps, 1))
    target = None
    for s in range(1, len(states)):
        if any(a[1] != b[1] for a, b in zip(states[s - 1], states[s])):
            target = s - 1          # decode step index whose seal is timed
            break
    if w.bulk_seal_step >= 0:
        target = ("bulk", w.bulk_seal_step)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    after = None
    if target is None:
        # no seal in the measured steps: append up to 32 more groups per sequence and layer
        # (seeded synthetic rows) and time one seal of them over all layers
        groups = bulk_seal_prefill(w, cache, ds, seq_ids, stream)
        torch.cuda.synchronize()
        ev0.record()
        groups = _lib.kv_seal(cache.h, -1, seq_ids, w.keep, stream)
        ev1.record()
        torch.cuda.synchronize()
        t = ev0.elapsed_time(ev1) / 1e3
        kind = "bulk seal of appended groups, all layers, one launch"
    elif isinstance(target, tuple):
        for s in range(target[1]):
            _lib.kv_decode_step(cache.h, w.n_layers, seq_ids, inp.q[s].data_ptr(), inp.k[s].data_ptr(),
                                inp.v[s].data_ptr(), out.data_ptr(), -1, w.keep, cache.ws.data_ptr(),
                                cache.ws_bytes, None, stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("bulk_seal")
        ev0.record()
        groups = _lib.kv_seal(cache.h, -1, seq_ids, w.keep, stream)
        ev1.record()
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        t = ev0.elapsed_time(ev1) / 1e3
        kind = "bulk seal, all layers, one launch"
        after = decode_after(w, cache, inp, seq_ids, out, stream, target[1])
    else:
        for s in range(target):
            _lib.kv_decode_step(cache.h, w.n_layers, seq_ids, inp.q[s].data_ptr(), inp.k[s].data_ptr(),
                                inp.v[s].data_ptr(), out.data_ptr(), w.seal_trigger, w.keep, cache.ws.data_ptr(),
                                cache.ws_bytes, None, stream)
        for l in range(w.n_layers):
            _lib.kv_append(cache.h, l, seq_ids, 1, inp.k[target, l].data_ptr(), inp.v[target, l].data_ptr(), stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("policy_seal")
        ev0.record()
        groups = _lib.kv_seal(cache.h, -1, seq_ids, w.keep, stream)
        ev1.record()
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        t = ev0.elapsed_time(ev1) / 1e3
        kind = "seal at the policy's trigger, all layers in one call (as the decode step issues it)"
    from quantized_kv_cache_gb300.configs import record_bytes
    D, H = w.head_dim, w.n_kv_heads
    read = 128 * H * 2 * ((D // 128) * 98 if w.journal == "tq6_0" else D * 2)
    write = H * (record_bytes(w.k_body, D) + record_bytes(w.v_body, D))
    hbm, _ = peaks()
    gps = groups / t if t > 0 else None
    res = {"groups_per_s": round(gps, 1) if gps else None, "groups": groups, "seconds": round(t, 6),
           "bytes_per_group": read + write, "hbm_frac": round(gps * (read + write) / 1e9 / hbm, 4) if gps else None,
           "kind": kind, "group": "128 positions x 1 layer x all KV heads x K and V"}
    if w.k_body.startswith("kvarn") and gps:
        # KVarN's balancing is bound by fp32 arithmetic: the method's fp32 operations per value
        # (no fused multiply-adds in the codec) against the fp32 lanes' issue rate
        per_value = KVARN_OPS_PER_VALUE + (KVARN_ROT_OPS if w.journal != "tq6_0" else KVARN_TQ6_OPS)
        ops = gps * 128 * H * 2 * D * per_value
        res["alu"] = {"bound": "alu", "ops_per_value": per_value, "achieved_tops": round(ops / 1e12, 3),
                      "peak_tops": FP32_PEAK_TOPS, "frac": round(ops / 1e12 / FP32_PEAK_TOPS, 4),
                      "peak_source": "152 SMs x 128 fp32 lanes x 2,070 MHz, one operation per lane per cycle"}
    if after:
        res["decode_after_seal"] = after
    return res


def prefill_bytes(w, n0, S1):
    """Algorithmic bytes of one kv_prefill of n0 positions of one layer (all KV heads) from an
    empty sequence that ends with S1 sealed: the fp16 input read once; the sealed groups'
    records, the sink, the journal rows of the unsealed positions past the sink and the exact
    tail (a tq6_0 ring only) written once."""
    from quantized_kv_cache_gb300.configs import record_bytes
    H, D = w.n_kv_heads, w.head_dim
    rows = 2 * H                                              # K and V rows of all heads
    b = n0 * rows * 2 * D                                     # input
    b += (S1 - 128) // 128 * H * (record_bytes(w.k_body, D) + record_bytes(w.v_body, D))
    b += min(n0, 128) * rows * 2 * D                          # sink
    unsealed = max(0, n0 - max(S1, 128))
    if w.journal == "tq6_0":
        b += unsealed * rows * (D // 128) * 98 + min(unsealed, w.tail) * rows * 2 * D
    else:
        b += unsealed * rows * 2 * D
    return b


def measure_prefill(w, ds, seq_ids, stream, reps=3):
    """kv_prefill of every sequence's whole context into a fresh one-layer cache (the layers
    are independent and alike), one call per sequence, timed with CUDA events after an untimed
    run; the inputs are generated in HBM first. Positions/s count positions of one layer, all
    KV heads."""
    import torch
    import quantized_kv_cache_gb300 as pkg
    from quantized_kv_cache_gb300 import synth, _lib
    H, D = w.n_kv_heads, w.head_dim
    cfg = w.config(n_layers=1)
    cache = pkg.KVCache(cfg, ds.dev.index)
    bufs = []
    for seq in seq_ids:
        n0 = w.contexts[seq]
        k = torch.empty((1, n0, H, D), dtype=torch.float16, device=ds.dev)
        v = torch.empty_like(k)
        ds.kv(synth.T_K, 0, seq, 0, n0, k, stream)
        ds.kv(synth.T_V, 0, seq, 0, n0, v, stream)
        bufs.append((k, v))
    torch.cuda.synchronize()

    def run():
        g = 0
        for seq, (k, v) in zip(seq_ids, bufs):
            g += cache.prefill(0, [seq], k, v, w.keep, stream)
        return g

    def reset():
        for seq in seq_ids:
            _lib.kv_reset(cache.h, 0, seq)

    run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(reps):
        reset()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("prefill")
        e0.record()
        groups = run()
        e1.record()
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3)
    status = _lib.kv_get_status(cache.h)
    states = [cache.state(0, seq) for seq in seq_ids]
    cache.close()
    t = sorted(times)[len(times) // 2]
    pos = sum(w.contexts[s] for s in seq_ids)
    byts = sum(prefill_bytes(w, w.contexts[s], S) for s, (_, S) in zip(seq_ids, states))
    hbm, _ = peaks()
    res = {"positions_per_s": round(pos / t, 1), "positions": pos, "groups_sealed": groups,
           "seconds": round(t, 6), "algorithmic_bytes": byts, "achieved_gbs": round(byts / t / 1e9, 2),
           "hbm_frac": round(byts / t / 1e9 / hbm, 4), "status": status,
           "kind": "kv_prefill of each sequence's whole context (keep = the workload's), one layer, "
                   "one call per sequence, median of 3"}
    if w.k_body.startswith("kvarn"):
        per_value = KVARN_OPS_PER_VALUE + (KVARN_ROT_OPS if w.journal != "tq6_0" else KVARN_TQ6_OPS)
        ops = groups * 128 * H * 2 * D * per_value / t
        res["alu"] = {"bound": "alu", "ops_per_value": per_value, "achieved_tops": round(ops / 1e12, 3),
                      "peak_tops": FP32_PEAK_TOPS, "frac": round(ops / 1e12 / FP32_PEAK_TOPS, 4),
                      "note": "the sealed groups' balancing only"}
    return res


def decode_after(w, cache, inp, seq_ids, out, stream, s0, max_steps=16):
    """Decode throughput after the bulk seal (the headline steps run before it): the steps
    s0 .. of the same inputs, the first one untimed (the graph is rebuilt after the seal)."""
    import torch
    from quantized_kv_cache_gb300 import _lib
    n = min(max_steps, inp.q.shape[0] - s0)
    if n < 2:
        return None
    def run(s):
        _lib.kv_decode_step(cache.h, w.n_layers, seq_ids, inp.q[s].data_ptr(), inp.k[s].data_ptr(),
                            inp.v[s].data_ptr(), out.data_ptr(), w.seal_trigger, w.keep, cache.ws.data_ptr(),
                            cache.ws_bytes, None, stream)
    run(s0)
    torch.cuda.synchronize()
    # lengths before each timed step (no seal falls in them: the bulk-seal workload never seals
    # during decode), after its append
    st0 = [cache.state(0, q) for q in seq_ids]
    byts = sum(layer_step_bytes(w, [(N + 1 + i, S) for N, S in st0]) for i in range(n - 1)) * w.n_layers
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for s in range(s0 + 1, s0 + n):
        run(s)
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3
    hbm, _ = peaks()
    return {"value": round(byts / t / 1e9, 2), "unit": UNIT, "steps": n - 1, "ms_per_step": round(t / (n - 1) * 1e3, 4),
            "pct_of_hbm_peak": round(100 * byts / t / 1e9 / hbm, 2),
            "note": "decode steps after the bulk seal (all but the newest 4,096 positions of each sequence sealed)"}


def measure_e2e(w, cache, inp, seq_ids, out, stream, K, total_bytes, world):
    """The same K steps through kv_decode_step with host buffers: each step copies its q, k,
    v (all layers) from pinned host memory and copies the outputs back, inside the timing."""
    import torch
    from quantized_kv_cache_gb300 import _lib
    hq = inp.q[:K].cpu().pin_memory()
    hk = inp.k[:K].cpu().pin_memory()
    hv = inp.v[:K].cpu().pin_memory()
    hout = torch.empty((K,) + tuple(out.shape), dtype=out.dtype).pin_memory()
    dq, dk, dv = torch.empty_like(inp.q[0]), torch.empty_like(inp.k[0]), torch.empty_like(inp.v[0])
    torch.cuda.synchronize()
    dist_barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for s in range(K):
        dq.copy_(hq[s], non_blocking=True)
        dk.copy_(hk[s], non_blocking=True)
        dv.copy_(hv[s], non_blocking=True)
        _lib.kv_decode_step(cache.h, w.n_layers, seq_ids, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                            out.data_ptr(), w.seal_trigger, w.keep, cache.ws.data_ptr(), cache.ws_bytes, None, stream)
        hout[s].copy_(out, non_blocking=True)
    t1.record()
    torch.cuda.synchronize()
    dist_barrier(world)
    el = dist_max(t0.elapsed_time(t1) / 1e3, world)
    h2d = dq.numel() * 2 + dk.numel() * 2 + dv.numel() * 2
    return {"value": round(total_bytes * world / el / 1e9, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": out.numel() * 2, "ms_per_step": round(el / K * 1e3, 4)}


def config_block(w, K):
    D = w.head_dim
    per_step = layer_step_bytes(w, [(n + 1, S) for n, S in initial_states(w, w.contexts)]) * w.n_layers
    return {"workload": w.name, "layers": w.n_layers, "kv_heads": w.n_kv_heads, "head_dim": D,
            "q_heads": w.n_q_heads, "batch": len(w.contexts), "contexts": w.contexts,
            "body": f"{w.k_body}/{w.v_body}", "journal": w.journal, "tail": w.tail, "decode_steps": K,
            "seal": f"keep {w.keep}, trigger {w.seal_trigger}",
            "l2": f"inputs larger than L2: each step reads ~{per_step / 1e6:.0f} MB of cache (L2 129 MB)",
            "inputs": "seeded synthetic fp16 K/V/q (splitmix64 counter streams over a normal quantile table)"}


# --------------------------------------------------------------------------- oracle arm
def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k = line.split(":")[0].strip().lower()
                if k in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
        # Arm: no model name line; report the implementer / part numbers
        with open("/proc/cpuinfo") as f:
            parts = {l.split(":")[0].strip(): l.split(":", 1)[1].strip() for l in f if ":" in l}
        if "CPU part" in parts:
            # Arm's part numbers of its Neoverse cores (implementer 0x41)
            names = {"0xd0c": "Neoverse N1", "0xd40": "Neoverse V1", "0xd49": "Neoverse N2", "0xd4f": "Neoverse V2"}
            part = parts["CPU part"]
            name = names.get(part, "") if parts.get("CPU implementer") == "0x41" else ""
            return f"{name + ' ' if name else ''}(implementer {parts.get('CPU implementer', '?')} part {part})"
    except Exception:
        pass
    return "unknown"


def cpu_baseline(workload, steps=4):
    """Time the oracle in a fresh process that spreads the sample over the host's cores."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-sample", workload, str(steps)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=1800)
    if r.returncode != 0:
        return {"value": None, "unit": UNIT, "cores": host_cores(), "kind": "oracle", "error": r.stderr[-400:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def oracle_units(w, steps, cores):
    """Independent units of the oracle sample: (KV head, first step, end step) of layer 0 of
    sequence 0. Each KV head's steps run in order (a step appends before it attends), so a
    unit replays the steps before its range untimed; ranges split each head's steps so that
    there are about as many units as cores."""
    heads = w.n_kv_heads
    per_head = max(1, min(steps, cores // heads if cores >= heads else 1))
    units = []
    for h in range(heads):
        for i in range(per_head):
            s0, s1 = steps * i // per_head, steps * (i + 1) // per_head
            if s1 > s0:
                units.append((h, s0, s1))
    return units


def _oracle_unit(workload, head, s0, s1, barrier, queue):
    """One unit: the oracle cache of (layer 0, sequence 0, head) built from the synthetic
    inputs and advanced to step s0, plus one warm-up attention (not timed), then steps s0 ..
    s1 - 1 timed: append, seal by the policy, dequantize every region and the fp64 attention
    of the head's query group."""
    import numpy as np
    from quantized_kv_cache_gb300 import configs, synth
    from quantized_kv_cache_gb300.runner import prefill_plan
    from oracle import attention
    from oracle.cache import HeadCache, HeadConfig
    try:
        w = configs.WORKLOADS[workload]
        n0, D, G = w.contexts[0], w.head_dim, w.G
        hc = HeadCache(HeadConfig(D, w.k_body, w.v_body, w.journal, w.tail_fmt, w.tail, w.ring))
        tb = time.time()
        pos = 0
        for c, seal in prefill_plan(w, n0):
            hc.append(synth.kv_values(w.seed, synth.T_K, 0, 0, head, pos, c, D, w.n_out, w.out_factor),
                      synth.kv_values(w.seed, synth.T_V, 0, 0, head, pos, c, D))
            pos += c
            if seal:
                hc.seal(w.keep)

        def advance(s):
            hc.append(synth.kv_values(w.seed, synth.T_K, 0, 0, head, n0 + s, 1, D, w.n_out, w.out_factor),
                      synth.kv_values(w.seed, synth.T_V, 0, 0, head, n0 + s, 1, D))
            if configs.should_seal(w, hc.N, hc.S):
                hc.seal(w.keep)

        for s in range(s0):
            advance(s)
        # one untimed attention over the current cache first (the process's first pass pays
        # its page faults and imports)
        q = synth.q_values(w.seed, 0, 0, s0, w.n_q_heads, D)
        attention.attend(q[head * G:(head + 1) * G].astype(np.float64), hc.regions(), hc.cfg.rot, 1 / np.sqrt(D))
        t_build = time.time() - tb
        barrier.wait()
        t0 = time.time()
        nbytes = 0
        for s in range(s0, s1):
            q = synth.q_values(w.seed, 0, 0, s, w.n_q_heads, D)
            advance(s)
            attention.attend(q[head * G:(head + 1) * G].astype(np.float64), hc.regions(), hc.cfg.rot,
                             1 / np.sqrt(D))
            nbytes += (layer_step_bytes(w, [(hc.N, hc.S)]) - 2 * w.n_q_heads * D * 2) // w.n_kv_heads \
                + 2 * G * D * 2
        queue.put((nbytes, t0, time.time(), t_build, None))
    except Exception as e:   # reported by the parent
        try:
            barrier.abort()
        except Exception:
            pass
        queue.put((0, 0.0, 0.0, 0.0, repr(e)))


def oracle_sample(workload, steps):
    """The oracle's decode attention of layer 0 of sequence 0 over `steps` steps and every KV
    head, as independent units in spawned single-threaded processes (one per core at most),
    timed from a common start after every unit has built its cache."""
    import multiprocessing as mp
    from quantized_kv_cache_gb300 import configs
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    w = configs.WORKLOADS[workload]
    cores = host_cores()
    units = oracle_units(w, steps, cores)
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(len(units))
    queue = ctx.Queue()
    procs = [ctx.Process(target=_oracle_unit, args=(workload, h, s0, s1, barrier, queue)) for h, s0, s1 in units]
    for p in procs:
        p.start()
    try:
        res = [queue.get(timeout=1500) for _ in procs]
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    errs = [r[4] for r in res if r[4]]
    if errs:
        raise RuntimeError(errs[0])
    nbytes = sum(r[0] for r in res)
    t0, t1 = min(r[1] for r in res), max(r[2] for r in res)
    return {"value": round(nbytes / (t1 - t0) / 1e9, 6), "unit": UNIT, "cores": len(units), "kind": "oracle",
            "host_cores": cores, "cpu_model": cpu_model(),
            "sample": f"{workload}: layer 0, sequence 0, {w.n_kv_heads} of {w.n_kv_heads} KV heads, {steps} "
                      f"decode step(s) at {w.contexts[0]} positions (append, seal policy, dequantize every "
                      f"region, fp64 attention), as {len(units)} independent (head, step range) units in "
                      f"single-threaded processes; cache builds ({max(r[3] for r in res):.1f} s) not counted",
            "seconds": round(t1 - t0, 3)}


def run_reference(args, rank, world):
    """--impl reference: the oracle, timed on the host cores, on bounded samples."""
    if rank != 0:
        return None
    from quantized_kv_cache_gb300 import configs
    w = configs.WORKLOADS[args.workload]
    n = max(1, min(args.warmup + args.steps, 64))
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-sample", args.workload, str(n)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=3000)
    if r.returncode != 0:
        return {"impl": "reference", "unavailable": "oracle run failed: " + r.stderr.strip().splitlines()[-1][:200]}
    cb = json.loads(r.stdout.strip().splitlines()[-1])
    v = cb["value"]
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(cb["seconds"] / n * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(w, args.steps),
            "cpu_baseline": cb,
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "note": f"oracle timed on {n} decode step(s) of one layer (all KV heads of sequence 0, spread over "
                    f"{cb['cores']} cores); see cpu_baseline.sample"}


# --------------------------------------------------------------------------- distributed
def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("KVQ_BENCH_BACKEND", "nccl")
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def weak_value(bytes_per_rank, elapsed_max, world):
    """Whole-job GB/s under weak scaling: every rank reads bytes_per_rank; the job's time is the
    slowest rank's."""
    return bytes_per_rank * world / elapsed_max / 1e9


def dist_max(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    if len(sys.argv) > 1 and sys.argv[1] == "--oracle-sample":
        print(json.dumps(oracle_sample(sys.argv[2], int(sys.argv[3]))))
        return 0
    args = parse()
    rank, world, local = dist_init()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
