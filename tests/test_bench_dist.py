"""The N > 1 path of bench.py on CPU: two gloo ranks (127.0.0.1) run the bench's own
rendezvous, barrier and max-over-ranks helpers, the weak-scaling aggregation, and the reference
arm's rank filter (ranks other than 0 do no work and print nothing)."""

import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), KVQ_BENCH_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, _ = bench.dist_init()
    bench.dist_barrier(w)
    elapsed = 0.5 + 0.25 * r                      # rank 1 is the slow one
    emax = bench.dist_max(elapsed, w)
    value = bench.weak_value(1e9, emax, w)
    args = type("A", (), {"workload": "tiny_tbq4", "steps": 1, "warmup": 0})()
    ref = bench.run_reference(args, r, w) if r != 0 else "skipped"
    bench.dist_barrier(w)
    dist.destroy_process_group()
    q.put((r, w, emax, value, ref))


def test_two_gloo_ranks_share_max_time_and_weak_value():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    for r, w, emax, value, ref in out:
        assert w == world
        assert emax == pytest.approx(0.75)                  # max over ranks, seen by every rank
        assert value == pytest.approx(1e9 * 2 / 0.75 / 1e9)  # whole-job bytes / slowest rank's time
    assert out[1][4] is None                                # rank 1: the reference arm does nothing


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_max(1.25, 1) == 1.25
    assert bench.weak_value(2e9, 0.5, 1) == pytest.approx(4.0)


def test_oracle_units_cover_every_head_step_once():
    # the reference arm's units: every (KV head, step) of the sample exactly once, in ranges
    # that a unit can replay in order, and no more units than cores (or KV heads)
    sys.path.insert(0, ROOT)
    import bench
    from quantized_kv_cache_gb300 import configs
    for name in ("longctx_tbq4", "fa14b_q8q4", "hybrid27b_kvarn44"):
        w = configs.WORKLOADS[name]
        for steps, cores in [(1, 16), (4, 16), (25, 16), (3, 2), (64, 8), (2, 72)]:
            units = bench.oracle_units(w, steps, cores)
            seen = sorted((h, s) for h, s0, s1 in units for s in range(s0, s1))
            assert seen == [(h, s) for h in range(w.n_kv_heads) for s in range(steps)]
            assert len(units) <= max(cores, w.n_kv_heads)
            assert all(s1 > s0 for _, s0, s1 in units)
