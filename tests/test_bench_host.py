"""Host logic of bench.py: the multi-rank aggregation (max of the step time,
sum of the work) over two gloo ranks on the CPU, and the scored-key byte
accounting against the oracle's cache geometry."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

import bench
import synth


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), HD_BENCH_BACKEND="gloo")
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(world)
    t, u = bench.reduce_timing(10.0 + rank, 100.0 * (rank + 1), world, None)
    queue.put((rank, t, u))
    bench.barrier(world)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_reduce_timing_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results == [(0, 11.0, 300.0), (1, 11.0, 300.0)]


def test_scored_keys_match_the_oracle_cache_geometry(orc):
    c = np.array([0, 1, 200, 510, 511, 512, 513, 4096, 32768], np.int32)
    for layout in (synth.LAYOUT_RING, synth.LAYOUT_ROLL):
        got = bench.scored_keys(synth.SLIDING, c, layout)
        cached = np.array([orc.cache_len(synth.SLIDING, layout, 512, int(x)) for x in c])
        # the new entry is scored too; a full roll window drops its oldest entry first
        want = cached + 1 - ((layout == synth.LAYOUT_ROLL) & (cached == 512))
        assert np.array_equal(got, want), layout
    full = bench.scored_keys(synth.FULL, c, synth.LAYOUT_RING)
    assert np.array_equal(full, np.array([orc.cache_len(synth.FULL, 0, 512, int(x)) + 1 for x in c]))


def test_step_bytes_of_the_4k_step_match_the_footprint_model(orc):
    """At batch 1, context 4096, the ring step scores every cached entry plus the
    new one: the footprint of the page's kv_cache_bytes plus one entry per layer."""
    c = np.array([4096], np.int32)
    hybrid, _ = orc.kv_cache_bytes(synth.SPARK_LAYER_TYPES, synth.LAYOUT_RING, 512, 2, 256, 4096)
    assert bench.step_bytes(synth.SPARK_LAYER_TYPES, c, 2, synth.LAYOUT_RING) == hybrid + 28 * 2048


def test_step_plan_of_the_benchmark_workloads():
    """The chunk plan and CTA count bench.py reports for its step grids (152 SMs)."""
    import synth as s
    assert bench.step_plan(s.SPARK_LAYER_TYPES, 64, 2, 4, 32679, s.LAYOUT_RING, "bf16", 152) == \
        {"chunk_keys": 2048, "grid_ctas": 17024}
    assert bench.step_plan(s.SPARK_LAYER_TYPES, 1, 2, 4, 4096, s.LAYOUT_RING, "bf16", 152) == \
        {"chunk_keys": 640, "grid_ctas": 140}
    # rolled windows take one chunk per sequence whatever the chunk size
    roll = bench.step_plan(s.SPARK_LAYER_TYPES, 1, 2, 4, 4096, s.LAYOUT_ROLL, "bf16", 152)
    assert roll["grid_ctas"] == 2 * (21 * 1 + 7 * -(-4096 // roll["chunk_keys"]))
