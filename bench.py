"""Benchmark of the hybrid decode-attention step on GB300.

Workload (default): the 28-layer step ([sliding x3, full] x7, Spark-X2.5
shape from vllm_omni/edge/spark_export.py) at batch 64 with per-sequence
contexts uniform in [512, 32768], 8 q / 2 kv heads, head_dim 256, bf16 KV
contiguous per sequence with a lengths array, sink fp32 N(0,1).  One step =
rope_append_kv + attention for every layer, through decode_step.

Metric: KV-read HBM GB/s = scored-key bytes per step / step time, where a
scored key costs one bf16 K row and one bf16 V row per kv head (1024 B at
head_dim 256); sliding layers score min(c, 511) + 1 keys, full layers c + 1.
The line also gives us per step, the roofline of the dominant kernel (the
full-layer split-K pass), the oracle timed on the host cores, an end-to-end
figure with host buffers, the same step with the per-head output gate, and the
batch-1 28-layer step as a secondary figure.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Multi-GPU (torchrun, one rank per GPU): every rank runs the same per-GPU
workload on its own sequences (weak scaling, no data-path collective); the
step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

KV_ROW_BYTES = 2 * synth.HEAD_DIM * 2       # K row + V row, bf16, one kv head
FP8_ROW_BYTES = 2 * synth.HEAD_DIM          # K row + V row, E4M3 codes, one kv head
DEFAULT_WORKLOAD = "step28_b64_c512_32768"
SECONDARY_WORKLOAD = "step28_b1_c4096"
METRIC = "KV-read HBM GB/s (% of GB300 peak); µs per 28-layer decode step"
# ncu DRAM-byte captures on the small block4_b16 case (about 1.2 GB on the device,
# larger than L2): DRAM bytes per algorithmic byte, scaled to a launch of the
# benchmarked workload (the kernels read every K/V row once, so traffic grows with
# the scored keys).
PROFILE_SUMMARY = {"step": os.path.join(ROOT, "profiles", "attn_step_grid_block4_b16_traffic.txt"),
                   "full": os.path.join(ROOT, "profiles", "attn_layer_kernel_full_block4_b16_traffic.txt")}


# ------------------------------------------------------------------ helpers --

def scored_keys(layer_type: int, context: np.ndarray, layout: int) -> np.ndarray:
    if layer_type == synth.FULL:
        return context.astype(np.int64) + 1
    keep = synth.WINDOW - 1 if layout != synth.LAYOUT_ROLL else synth.WINDOW
    if layout == synth.LAYOUT_ROLL:
        return np.minimum(context.astype(np.int64) + 1, keep)
    return np.minimum(context.astype(np.int64), keep) + 1


def step_bytes(types, context, num_kv_heads, layout, row_bytes=KV_ROW_BYTES) -> int:
    return int(sum(scored_keys(t, context, layout).sum() for t in types) * num_kv_heads * row_bytes)


def step_plan(types, batch, num_kv_heads, group, max_ctx, layout, kv, num_sms) -> dict:
    """The step grid's chunk plan for a single-token step (hd_plan_step_split, the
    model decode_step uses) and the CTA count it gives."""
    import full_gqa_decode_gb300 as hd
    roll = layout == synth.LAYOUT_ROLL
    keys = [max_ctx if t == synth.FULL else (synth.WINDOW - 1) for t in types]
    one = [roll and t == synth.SLIDING for t in types]
    c = hd.hd_plan_step_split(keys, batch, num_kv_heads, group, num_sms,
                              kv_dtype=hd.HD_KV_FP8_E4M3 if kv == "fp8" else hd.HD_KV_BF16, one_chunk=one)
    ctas = sum(batch * num_kv_heads * (1 if o else max(1, -(-k // c))) for k, o in zip(keys, one))
    return {"chunk_keys": c, "grid_ctas": ctas}


def describe_layers(types) -> str:
    n_full = sum(1 for t in types if t == synth.FULL)
    if list(types) == synth.SPARK_LAYER_TYPES:
        return f"{len(types)} = [sliding x3, full] x7"
    return f"{len(types)} ({len(types) - n_full} sliding, {n_full} full)"


def describe_lengths(recipe) -> str:
    kind = recipe[0]
    if kind == "fixed":
        return f"{recipe[1]} for every sequence"
    if kind == "uniform":
        return f"uniform [{recipe[1]}, {recipe[2]}] per sequence"
    if kind == "mixed":
        return f"{recipe[1]}, with {recipe[2]:.0%} of sequences uniform in [1, {recipe[3]}]"
    return str(recipe)


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("attn_kernel.cuh", "hd_internal.h", "rope_round.cuh", "e4m3.cuh"):
        with open(os.path.join(ROOT, "full_gqa_decode_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kind: str, algorithmic_bytes: int):
    """DRAM bytes per launch of the step grid ("step") or of the full-layer kernel
    ("full") for a launch of `algorithmic_bytes` scored-KV bytes: the committed ncu
    summary's DRAM bytes per algorithmic byte (small case) times those bytes.  None
    when the summary is absent or the kernel changed since it was taken."""
    path = PROFILE_SUMMARY[kind]
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    if kv.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return round(float(kv["dram_bytes_per_algorithmic_byte"]) * algorithmic_bytes)
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        import torch
        self.proc = None
        try:
            self.gpu = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            self.gpu = str(device.index)
        self.path = os.path.join(tempfile.gettempdir(), f"hd_bench_clocks_dev{device.index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            self.proc.wait(timeout=5)
            self.fh.close()

    def summary(self) -> dict:
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------- distributed plumbing --

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("HD_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def reduce_timing(elapsed_ms: float, units: float, world: int, device=None) -> tuple[float, float]:
    """Max of the step time over ranks and the sum of the work units over ranks."""
    if world == 1:
        return elapsed_ms, units
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ------------------------------------------------------------- the workload --

class Workload:
    """Device-resident inputs of one workload (caches, per-layer q/k/v, outputs)."""

    def __init__(self, name: str, device, seed: int = 0, layout: int = synth.LAYOUT_AUTO, kv: str = "bf16",
                 tokens: int = 1):
        import torch
        import full_gqa_decode_gb300 as hd
        spec = synth.WORKLOADS[name]
        self.name, self.spec, self.layout, self.kv, self.tokens = name, spec, layout, kv, tokens
        tq = (tokens,) if tokens > 1 else ()   # token index of a multi-token step
        fp8 = kv == "fp8"
        self.row_bytes = FP8_ROW_BYTES if fp8 else KV_ROW_BYTES
        self.types = list(spec["layer_types"])
        self.B, self.Hq, self.Hkv = spec["batch"], spec["num_q_heads"], spec["num_kv_heads"]
        D = synth.HEAD_DIM
        rng = synth.generator(seed)
        self.context = synth.context_lengths(rng, spec["lengths"], self.B)
        self.max_ctx = int(self.context.max())
        sink = synth.sink_vector(rng, spec["sink"], self.Hq)
        self.cfg = hd.Config(layer_types=self.types, num_q_heads=self.Hq, num_kv_heads=self.Hkv,
                             cache_layout=layout, max_batch=self.B, max_context=self.max_ctx + tokens - 1,
                             kv_dtype=hd.HD_KV_FP8_E4M3 if fp8 else hd.HD_KV_BF16)
        self.ctx = hd.hybrid_decode_init(self.cfg)
        self.context_d = torch.from_numpy(self.context).to(device)
        self.sink = None if sink is None else sink.to(device)
        ring = layout != synth.LAYOUT_ROLL
        self.layers, self.io, self.io_gated = [], [], []
        # every layer's q, k, v (and out, lse) are slices of one buffer each, so a
        # step's inputs move host -> device in one copy (and its outputs back in two)
        per_q, per_kv = self.B * tokens * self.Hq * D, self.B * tokens * self.Hkv * D
        nl = len(self.types)
        self.qkv = torch.empty(nl, per_q + 2 * per_kv, dtype=torch.bfloat16, device=device)
        self.outs = torch.empty(nl, per_q, dtype=torch.bfloat16, device=device)
        self.lses = torch.empty(nl, self.B * tokens * self.Hq, dtype=torch.float32, device=device)
        for i, t in enumerate(self.types):
            cap = (synth.WINDOW - 1 if ring else synth.WINDOW) if t == synth.SLIDING else self.max_ctx + tokens
            kc = torch.empty(self.B, self.Hkv, cap, D, dtype=torch.uint8 if fp8 else torch.bfloat16, device=device)
            vc = torch.empty_like(kc)
            if fp8:  # per-layer, per-kv-head scales; codes of N(0,1) / scale
                ks, vs = synth.kv_scales(rng, self.Hkv).to(device), synth.kv_scales(rng, self.Hkv).to(device)
                synth.cuda_e4m3_codes_(kc, ks, seed * 1000 + 2 * i + 1)
                synth.cuda_e4m3_codes_(vc, vs, seed * 1000 + 2 * i + 2)
            else:
                ks = vs = None
                synth.cuda_normal_bf16_(kc, seed * 1000 + 2 * i + 1)
                synth.cuda_normal_bf16_(vc, seed * 1000 + 2 * i + 2)
            g = torch.Generator(device=device)
            g.manual_seed(seed * 1000 + 500 + i)
            q = self.qkv[i, :per_q].view(self.B, *tq, self.Hq, D)
            k = self.qkv[i, per_q:per_q + per_kv].view(self.B, *tq, self.Hkv, D)
            v = self.qkv[i, per_q + per_kv:].view(self.B, *tq, self.Hkv, D)
            for x in (q, k, v):
                x.copy_(torch.randn(x.shape, generator=g, device=device))
            out = self.outs[i].view(self.B, *tq, self.Hq, D)
            lse = self.lses[i].view(self.B, *tq, self.Hq)
            cache = hd.kv_cache(kc, vc, ks, vs)
            self.layers.append(dict(q=q, k=k, v=v, kc=kc, vc=vc, out=out, lse=lse, cache=cache,
                                    k_scale=ks, v_scale=vs))
            self.io.append(hd.layer_io(q, k, v, cache, self.sink, out, lse))
            # per-step output-gate logits N(0, 1) for the gated variant of the step
            gate = torch.randn(self.B, *tq, self.Hq, generator=g, device=device)
            self.layers[-1]["gate"] = gate
            self.io_gated.append(hd.layer_io(q, k, v, cache, self.sink, out, lse, gate=gate))
        self.io_arr = hd.layer_array(self.ctx, self.io)              # built once, passed every step
        self.io_gated_arr = hd.layer_array(self.ctx, self.io_gated)
        self.bytes = step_bytes(self.types, self.context, self.Hkv, layout, self.row_bytes)
        full_idx = [i for i, t in enumerate(self.types) if t == synth.FULL]
        self.full_layer_bytes = (int(scored_keys(synth.FULL, self.context, layout).sum()) * self.Hkv
                                 * self.row_bytes) if full_idx else 0
        self.sliding_layer_bytes = (int(scored_keys(synth.SLIDING, self.context, layout).sum()) * self.Hkv
                                    * self.row_bytes)

    def step(self, stream=None, gated=False):
        import full_gqa_decode_gb300 as hd
        io = self.io_gated_arr if gated else self.io_arr
        if self.tokens > 1:
            hd.decode_step_tokens(self.ctx, self.context_d, io, self.B, self.tokens, self.max_ctx, stream)
        else:
            hd.decode_step(self.ctx, self.context_d, io, self.B, self.max_ctx, stream)

    def token_pass_bytes(self) -> int:
        """Scored-KV bytes a multi-token step reads: the tokens of a sequence run in
        passes of up to 32 query rows with bf16 caches (16 with E4M3) and 8 tokens per
        kv head, each pass scoring the cache at context + first token of the pass
        (earlier passes' entries included)."""
        rows = 16 if self.kv == "fp8" else 32
        tmax, passes, t0 = min(8, max(1, rows // (self.Hq // self.Hkv))), [], 0
        while t0 < self.tokens:
            tp = 1
            while 2 * tp <= tmax and 2 * tp <= self.tokens - t0:
                tp *= 2
            passes.append(t0)
            t0 += tp
        total = 0
        for t0 in passes:
            ctx = self.context + t0
            for t in self.types:
                keys = ctx if t == synth.FULL else np.minimum(ctx, synth.WINDOW - 1)
                total += int(keys.sum()) * self.Hkv * self.row_bytes
        return total


def time_steps(run, steps: int, warmup: int, world: int, device) -> float:
    """ms per step over `steps` steps (after `warmup`), CUDA events on the current stream."""
    import torch
    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    barrier(world, device)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        run()
    end.record()
    torch.cuda.synchronize()
    barrier(world, device)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


# ------------------------------------------------------------- CPU baseline --

def oracle_sample(layer_caches, context, types, Hq, Hkv, sink, rng, threads, layout=synth.LAYOUT_RING):
    """Times the oracle on one [S,S,S,F] block of the step for the given sequences.
    layer_caches: per layer (kc, vc) uint16 arrays [B, Hkv, cap, D], or (kc, vc, k_scale,
    v_scale) with uint8 E4M3 codes. Returns (seconds, bytes)."""
    import oracle
    orc = oracle.load()
    D = synth.HEAD_DIM
    B = len(context)
    jobs = []
    for li, t in enumerate(types):
        rot, theta = synth.ROPE[t]
        kc, vc = layer_caches[li][:2]
        scales = {}
        if kc.dtype == np.uint8:
            scales = dict(k_scale=layer_caches[li][2], v_scale=layer_caches[li][3])
        for b in range(B):
            q = synth.bits(synth.normal_bf16(rng, (1, Hq, D)))
            k = synth.bits(synth.normal_bf16(rng, (1, Hkv, D)))
            v = synth.bits(synth.normal_bf16(rng, (1, Hkv, D)))
            jobs.append(dict(layer_type=t, layout=layout, window=synth.WINDOW, rotary_dim=rot,
                             rope_theta=theta, context=context[b:b + 1], q=q, k=k, v=v,
                             kcache=np.ascontiguousarray(kc[b:b + 1]), vcache=np.ascontiguousarray(vc[b:b + 1]),
                             sink=sink, **scales))
    row = FP8_ROW_BYTES if layer_caches[0][0].dtype == np.uint8 else KV_ROW_BYTES
    nbytes = step_bytes(types, context, Hkv, layout, row)
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(threads) as ex:   # ctypes releases the GIL in the oracle
        list(ex.map(lambda j: orc.decode_layer(**j), jobs))
    return time.perf_counter() - t0, nbytes


def host_block_caches(spec, context, rng):
    """Host-generated caches of one [S,S,S,F] block (for the reference arm)."""
    B, Hkv, D = len(context), spec["num_kv_heads"], synth.HEAD_DIM
    out = []
    for t in [synth.SLIDING, synth.SLIDING, synth.SLIDING, synth.FULL]:
        cap = synth.WINDOW - 1 if t == synth.SLIDING else int(context.max()) + 1
        kc = np.empty((B, Hkv, cap, D), np.uint16)
        vc = np.empty_like(kc)
        for b in range(B):
            n = min(int(context[b]), cap)
            kc[b] = 0x7FC0
            vc[b] = 0x7FC0
            kc[b, :, :n] = synth.bits(synth.normal_bf16(rng, (Hkv, n, D)))
            vc[b, :, :n] = synth.bits(synth.normal_bf16(rng, (Hkv, n, D)))
        out.append((kc, vc))
    return out


def cpu_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


# ----------------------------------------------------------------- the arms --

def workload_config(spec, name, context, layout_name, kv, world) -> dict:
    """The `config` object of the JSON line, the same for both arms."""
    types = list(spec["layer_types"])
    layout = synth.LAYOUT_ROLL if layout_name == "roll" else synth.LAYOUT_RING
    row = FP8_ROW_BYTES if kv == "fp8" else KV_ROW_BYTES
    B = len(context)
    return {"workload": name, "global_batch": B * world, "per_gpu_batch": B,
            "layers": describe_layers(types), "heads": f"{spec['num_q_heads']} q / {spec['num_kv_heads']} kv",
            "head_dim": synth.HEAD_DIM, "contexts": describe_lengths(spec["lengths"]),
            "max_context": int(context.max()),
            "kv_bytes_per_step": step_bytes(types, context, spec["num_kv_heads"], layout, row),
            "sliding_layout": layout_name, "kv_dtype": kv,
            "l2": "inputs larger than L2 (no flush)", "parallelism": f"dp{world}"}


def run_reference(args, world, rank) -> int:
    """The oracle, as it stands, on the host cores: each step is a bounded sample
    (one [S,S,S,F] block of the step over every sequence).  ms_per_step is the
    timed block's own time; the whole 28-layer step at the same rate is given
    apart as ms_per_step_extrapolated."""
    if rank != 0:
        return 0
    spec = synth.WORKLOADS[args.workload]
    rng = synth.generator(0)
    context = synth.context_lengths(rng, spec["lengths"], spec["batch"])
    sink = synth.sink_vector(rng, spec["sink"], spec["num_q_heads"])
    sink = None if sink is None else sink.numpy()
    caches = host_block_caches(spec, context, rng)
    threads = cpu_threads()
    block = [synth.SLIDING, synth.SLIDING, synth.SLIDING, synth.FULL]
    for _ in range(args.warmup):
        oracle_sample(caches, context, block, spec["num_q_heads"], spec["num_kv_heads"], sink, rng, threads)
    secs, nbytes = 0.0, 0
    for _ in range(args.steps):
        s, n = oracle_sample(caches, context, block, spec["num_q_heads"], spec["num_kv_heads"], sink, rng,
                             threads)
        secs += s
        nbytes += n
    gbs = nbytes / secs / 1e9
    config = workload_config(spec, args.workload, context, "ring", "bf16", world)
    sample = (f"one [sliding x3, full] block of the 28-layer step over all {len(context)} sequences "
              f"({nbytes // args.steps / 1e9:.2f} GB of scored KV per step, caches drawn on the host "
              f"from the same recipe); fp64 oracle, {threads} host threads")
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs / args.steps * 1e3, 3),
            "ms_per_step_extrapolated": round(config["kv_bytes_per_step"] / (gbs * 1e9) * 1e3, 3),
            "ms_per_step_note": "ms_per_step times the sampled [sliding x3, full] block; "
                                "ms_per_step_extrapolated is the whole 28-layer step at the same GB/s",
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config,
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, world, rank, local) -> int:
    import torch
    import full_gqa_decode_gb300 as hd
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    peaks = measured_peaks()
    layout = synth.LAYOUT_ROLL if args.layout == "roll" else synth.LAYOUT_RING
    wl = Workload(args.workload, device, seed=rank, layout=layout, kv=args.kv, tokens=args.tokens)
    # KV bytes a step reads: the scored keys, or with several tokens per sequence
    # every pass's read of the cache
    step_kv = wl.token_pass_bytes() if args.tokens > 1 else wl.bytes
    consumer = {"tensor-core": hd.HD_CONSUMER_TENSOR_CORE, "cuda-core": hd.HD_CONSUMER_CUDA_CORE,
                "tensor-memory": hd.HD_CONSUMER_TENSOR_MEMORY}[args.consumer]
    tensor = consumer != hd.HD_CONSUMER_CUDA_CORE
    hd.hybrid_decode_set_consumer(wl.ctx, consumer)
    torch.cuda.synchronize()

    # device-resident timed region (W warm-up steps first, then exactly K timed steps).
    # With the tensor-core consumer every step is one step grid (the attention of all
    # layers), the dominant kernel, bracketed by events on its stream; the CUDA-core
    # consumer runs one kernel per layer, and the first full layer of every step is
    # bracketed (that launch alone runs without early start; the others overlap).
    fused = tensor and args.fusion == "on"
    hd.hybrid_decode_set_step_fusion(wl.ctx, fused)
    kind = hd.HD_PROFILE_KIND_STEP if fused else hd.HD_FULL
    hd.hybrid_decode_set_profiling(wl.ctx, hd.HD_PROFILE_STEP if fused else hd.HD_PROFILE_FULL | hd.HD_PROFILE_FIRST_ONLY)
    with ClockSampler(device) as clocks:
        for _ in range(args.warmup):
            wl.step()
        torch.cuda.synchronize()
        hd.hybrid_decode_profile(wl.ctx, kind)  # drop the warm-up records
        n0 = hd.hybrid_decode_launch_count(wl.ctx)
        ms = time_steps(wl.step, args.steps, 0, world, device)
        n1 = hd.hybrid_decode_launch_count(wl.ctx)
        dom_ms, dom_launches = hd.hybrid_decode_profile(wl.ctx, kind)
    hd.hybrid_decode_set_profiling(wl.ctx, 0)
    clk = clocks.summary()
    flags = hd.hybrid_decode_device_errors(wl.ctx)
    if flags:
        raise RuntimeError(f"device error flags {flags:#x} during the benchmark")
    ms_max, total_bytes = reduce_timing(ms, step_kv, world, device)
    gbs = total_bytes / (ms_max * 1e-3) / 1e9

    # diagnostic passes, outside the timed region: one kernel per layer, the first
    # full layer and every sliding layer bracketed alone
    layer_kernels = layer_kernel_rooflines(wl, peaks) if args.tokens == 1 else {}

    # roofline of the dominant kernel
    avg_ms = dom_ms / max(dom_launches, 1)
    per_launch = (step_kv * args.steps // max(dom_launches, 1)) if fused else wl.full_layer_bytes
    achieved = per_launch / (avg_ms * 1e-3) / 1e9 if dom_launches else None
    roofline = {"bound": "hbm", "achieved": round(achieved, 1) if achieved else None,
                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4) if achieved else None,
                "traffic": profiled_traffic("step" if fused else "full", per_launch),
                "traffic_source": "ncu DRAM read+write bytes per algorithmic byte on block4_b16_c512_32768 "
                                  "(profiles/), times this launch's algorithmic bytes",
                "kernel": (f"attn_layer_kernel step grid (the attention of all {len(wl.types)} layers); events "
                           f"around the grid of each timed step" if fused else
                           f"attn_layer_kernel, full layers ({args.consumer}); events around the first full "
                           f"layer of each timed step"),
                "algorithmic_bytes_per_launch": int(per_launch),
                "avg_launch_ms": round(avg_ms, 4), "launches": int(dom_launches), "peak_source": peaks["source"]}
    roofline.update(layer_kernels)

    read_peak = read_stream_probe(device)
    if read_peak and achieved:
        roofline["read_stream_probe_gbs"] = round(read_peak, 1)
        roofline["frac_of_read_stream"] = round(achieved / read_peak, 4)

    # end to end: host buffers, copies inside the timed region
    e2e = e2e_measure(wl, args, world, device)

    # the same step with the per-head output gate fused into every layer's epilogue,
    # against the ungated step timed the same way (no profiling events)
    plain_ms = time_steps(wl.step, args.steps, args.warmup, 1, device)
    gated_ms = time_steps(lambda: wl.step(gated=True), args.steps, args.warmup, 1, device)
    # the same step with one kernel per layer (early start on), and with every
    # layer in full stream order (no early start)
    hd.hybrid_decode_set_step_fusion(wl.ctx, False)
    per_layer_ms = time_steps(wl.step, args.steps, args.warmup, 1, device)
    hd.hybrid_decode_set_layer_overlap(wl.ctx, False)
    serial_ms = time_steps(wl.step, args.steps, args.warmup, 1, device)
    # the same stream-order step replayed from a CUDA graph (how a serving loop
    # launches a decode step): the launches no longer wait on the host
    serial_graph_ms = graph_steps(wl, args, device)
    hd.hybrid_decode_set_layer_overlap(wl.ctx, True)
    hd.hybrid_decode_set_step_fusion(wl.ctx, True)
    if hd.hybrid_decode_device_errors(wl.ctx):
        raise RuntimeError("device error flags during the gated step")

    result = None
    if rank == 0:
        fp8 = fp8_step(device, args, consumer, layout, plain_ms) if args.kv == "bf16" and args.secondary else None
        multi = (multi_token_steps(device, args, consumer, layout, plain_ms)
                 if args.kv == "bf16" and args.secondary and args.layout == "ring" and tensor
                 else None)
        cpu = cpu_baseline(wl, device)
        secondary = secondary_batch1(device, args, consumer) if args.secondary else None
        others = (baseline_configs(device, args, consumer, read_peak)
                  if args.secondary and args.kv == "bf16" and args.workload == DEFAULT_WORKLOAD
                  and tensor else None)
        result = {"metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world,
                  "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
                  "us_per_step": round(ms_max * 1e3, 1), "higher_is_better": True, "scaling": "weak",
                  "vs_baseline": None, "dtype": "bf16" if args.kv == "bf16" else "fp8_e4m3 KV, f16 MMA",
                  "data": "synthetic",
                  "frac_of_peak_hbm": round(gbs / peaks["hbm_gbs"], 4),
                  "config": workload_config(wl.spec, wl.name, wl.context, args.layout, args.kv, world),
                  "step_grid": step_plan(wl.types, wl.B, wl.Hkv, wl.Hq // wl.Hkv, wl.max_ctx, wl.layout,
                                         args.kv, torch.cuda.get_device_properties(device).multi_processor_count)
                  if fused else None,
                  "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                  "gpu_launches": int(n1 - n0), "clocks": clk}
        result["output_gate"] = {"ms_per_step": round(gated_ms, 4),
                                 "value": round(step_kv / (gated_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                                 "ungated_ms_per_step": round(plain_ms, 4),
                                 "overhead_vs_ungated": round(gated_ms / plain_ms - 1.0, 4)}
        result["kernel_per_layer"] = {
            "ms_per_step": round(per_layer_ms, 4), "value": round(step_kv / (per_layer_ms * 1e-3) / 1e9, 1),
            "unit": "GB/s", "note": "step fusion off: one kernel per layer, each starting while the previous drains"}
        result["layers_in_stream_order"] = {
            "ms_per_step": round(serial_ms, 4), "value": round(step_kv / (serial_ms * 1e-3) / 1e9, 1),
            "unit": "GB/s", "note": "step fusion off and no layer starts before the previous one is complete",
            "cuda_graph": {"ms_per_step": round(serial_graph_ms, 4),
                           "value": round(step_kv / (serial_graph_ms * 1e-3) / 1e9, 1), "unit": "GB/s"}}
        if args.tokens > 1:
            result["config"].update(tokens_per_sequence=args.tokens, kv_bytes_read_per_step=step_kv)
        if fp8:
            result["fp8_kv"] = fp8
        if multi:
            result["multi_token"] = multi
        if secondary:
            result["secondary"] = secondary
        if others:
            result["baseline_configs"] = others
        print(json.dumps(result), flush=True)
    return 0


def read_stream_probe(device, gib: int = 4):
    """GB/s of a pure TMA read stream over a fresh buffer (the library's probe),
    median of 5 passes after 2 warm-up passes; None if memory is short."""
    import torch
    import full_gqa_decode_gb300 as hd
    try:
        buf = torch.empty(gib << 30, dtype=torch.uint8, device=device)
    except torch.OutOfMemoryError:
        return None
    buf.fill_(1)
    for _ in range(2):
        hd.hybrid_decode_read_probe(buf)
    times, nbytes = [], 0
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        nbytes = hd.hybrid_decode_read_probe(buf)
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    del buf
    return nbytes / (statistics.median(times) * 1e-3) / 1e9


def layer_kernel_rooflines(wl, peaks) -> dict:
    """Outside the timed region, with step fusion off (one kernel per layer): the
    first full layer of each of 3 steps and every sliding layer, each launch
    bracketed by events alone; achieved GB/s over that layer's scored KV bytes."""
    import full_gqa_decode_gb300 as hd
    hd.hybrid_decode_set_step_fusion(wl.ctx, False)
    for _ in range(2):   # unbracketed: the layer kernels' first launches load their code
        wl.step()
    out = {}
    for name, mask, kind, nbytes in (("full_layers", hd.HD_PROFILE_FULL | hd.HD_PROFILE_FIRST_ONLY, hd.HD_FULL,
                                      wl.full_layer_bytes),
                                     ("sliding_layers", hd.HD_PROFILE_SLIDING, hd.HD_SLIDING,
                                      wl.sliding_layer_bytes)):
        hd.hybrid_decode_set_profiling(wl.ctx, mask)
        for _ in range(3):
            wl.step()
        t_ms, n = hd.hybrid_decode_profile(wl.ctx, kind)
        if n and nbytes:
            avg = t_ms / n
            gbs = nbytes / (avg * 1e-3) / 1e9
            out[name] = {"kernel": "attn_layer_kernel, one layer per launch", "achieved": round(gbs, 1),
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes_per_launch": nbytes,
                         "avg_launch_ms": round(avg, 4)}
    if "full_layers" in out:
        out["full_layers"]["traffic"] = profiled_traffic("full", wl.full_layer_bytes)
    hd.hybrid_decode_set_profiling(wl.ctx, 0)
    hd.hybrid_decode_set_step_fusion(wl.ctx, True)
    return out


def e2e_measure(wl, args, world, device) -> dict:
    """Same metric through the public API with pinned host buffers: every step copies
    that step's q/k/v (all layers, one buffer) and the contexts host->device, runs
    the step, and reads out and lse (all layers) back."""
    import torch
    host_in = wl.qkv.cpu().pin_memory()
    host_ctx = torch.from_numpy(wl.context).pin_memory()
    host_out = torch.empty_like(wl.outs, device="cpu").pin_memory()
    host_lse = torch.empty_like(wl.lses, device="cpu").pin_memory()
    h2d = host_in.numel() * host_in.element_size() + host_ctx.numel() * 4
    d2h = host_out.numel() * host_out.element_size() + host_lse.numel() * host_lse.element_size()

    def run():
        wl.context_d.copy_(host_ctx, non_blocking=True)
        wl.qkv.copy_(host_in, non_blocking=True)
        wl.step()
        host_out.copy_(wl.outs, non_blocking=True)
        host_lse.copy_(wl.lses, non_blocking=True)
    ms = time_steps(run, args.steps, args.warmup, world, device)
    ms_max, total = reduce_timing(ms, wl.token_pass_bytes() if wl.tokens > 1 else wl.bytes, world, device)
    return {"value": round(total / (ms_max * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(ms_max, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


def cpu_baseline(wl, device) -> dict:
    """The oracle on the host cores, on the first [S,S,S,F] block of this very
    workload (caches copied from the device before timing; compute only timed)."""
    block = list(range(4))
    caches = []
    for i in block:
        l = wl.layers[i]
        if wl.kv == "fp8":
            caches.append((synth.bits(l["kc"]), synth.bits(l["vc"]), l["k_scale"].cpu().numpy(),
                           l["v_scale"].cpu().numpy()))
        else:
            caches.append((synth.bits(l["kc"]), synth.bits(l["vc"])))
    sink = None if wl.sink is None else wl.sink.cpu().numpy()
    threads = cpu_threads()
    layout = synth.LAYOUT_ROLL if wl.layout == synth.LAYOUT_ROLL else synth.LAYOUT_RING
    secs, nbytes = 0.0, 0
    for rep in range(3):   # about 15 s of CPU work on 16 cores at the default workload
        s_, n_ = oracle_sample(caches, wl.context, [wl.types[i] for i in block], wl.Hq, wl.Hkv, sink,
                               synth.generator(99 + rep), threads, layout)
        secs, nbytes = secs + s_, nbytes + n_
    # one host thread on the first 8 sequences of the same block
    few = min(8, len(wl.context))
    secs1, nbytes1 = oracle_sample([tuple(x[:few] if x.ndim == 4 else x for x in c) for c in caches],
                                   wl.context[:few], [wl.types[i] for i in block], wl.Hq, wl.Hkv, sink,
                                   synth.generator(98), 1, layout)
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"layers 0-3 ([sliding x3, full]) of the step over all {len(wl.context)} sequences, "
                      f"three times: {nbytes / 1e9:.2f} GB scored KV, {secs:.1f} s on {threads} threads",
            "single_thread": {"value": round(nbytes1 / secs1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"the same block over the first {few} sequences, "
                                        f"{nbytes1 / 1e9:.2f} GB scored KV, {secs1:.1f} s"}}


def fp8_step(device, args, consumer, layout, bf16_ms) -> dict:
    """The same step with E4M3 caches (per-kv-head scales): step time, KV GB/s over
    the E4M3 bytes, and the full-layer kernel alone (events in a separate pass)."""
    import torch
    import full_gqa_decode_gb300 as hd
    wl = Workload(args.workload, device, seed=0, layout=layout, kv="fp8")
    hd.hybrid_decode_set_consumer(wl.ctx, consumer)
    ms = time_steps(wl.step, args.steps, args.warmup, 1, device)
    fused = consumer != hd.HD_CONSUMER_CUDA_CORE
    grid_ms, grid_n = 0.0, 0
    if fused:
        hd.hybrid_decode_set_profiling(wl.ctx, hd.HD_PROFILE_STEP)
        for _ in range(3):
            wl.step()
        grid_ms, grid_n = hd.hybrid_decode_profile(wl.ctx, hd.HD_PROFILE_KIND_STEP)
    hd.hybrid_decode_set_step_fusion(wl.ctx, False)
    for _ in range(2):   # unbracketed: the layer kernels' first launches load their code
        wl.step()
    hd.hybrid_decode_set_profiling(wl.ctx, hd.HD_PROFILE_FULL)
    for _ in range(3):
        wl.step()
    full_ms, full_n = hd.hybrid_decode_profile(wl.ctx, hd.HD_FULL)
    hd.hybrid_decode_set_profiling(wl.ctx, 0)
    hd.hybrid_decode_set_step_fusion(wl.ctx, True)
    flags = hd.hybrid_decode_device_errors(wl.ctx)
    if flags:
        raise RuntimeError(f"device error flags {flags:#x} in the FP8 step")
    peak = measured_peaks()["hbm_gbs"]
    res = {"ms_per_step": round(ms, 4), "us_per_step": round(ms * 1e3, 1),
           "value": round(wl.bytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "kv_bytes_per_step": wl.bytes,
           "speedup_vs_bf16_step": round(bf16_ms / ms, 3)}
    if grid_n:
        per_launch = wl.bytes * 3 // grid_n
        avg = grid_ms / grid_n
        res["step_grid"] = {"achieved": round(per_launch / (avg * 1e-3) / 1e9, 1), "unit": "GB/s",
                            "frac": round(per_launch / (avg * 1e-3) / 1e9 / peak, 4), "avg_launch_ms": round(avg, 4),
                            "algorithmic_bytes_per_launch": per_launch}
    if full_n:
        avg = full_ms / full_n
        res["full_layer_kernel"] = {"achieved": round(wl.full_layer_bytes / (avg * 1e-3) / 1e9, 1), "unit": "GB/s",
                                    "frac": round(wl.full_layer_bytes / (avg * 1e-3) / 1e9 / peak, 4),
                                    "avg_launch_ms": round(avg, 4),
                                    "algorithmic_bytes_per_launch": wl.full_layer_bytes}
    wl.ctx.close()
    del wl
    torch.cuda.empty_cache()
    return res


def multi_token_steps(device, args, consumer, layout, single_ms) -> list:
    """The same step decoding T = 2, 4 and 8 tokens per sequence (decode_step_tokens),
    against T single-token steps (the plain step time)."""
    import torch
    import full_gqa_decode_gb300 as hd
    res = []
    for T in (2, 4, 8):   # group 4: 8, 16 and 32 query rows per kv head (32: the tcgen05 pass)
        wl = Workload(args.workload, device, seed=0, layout=layout, tokens=T)
        hd.hybrid_decode_set_consumer(wl.ctx, consumer)
        ms = time_steps(wl.step, args.steps, args.warmup, 1, device)
        if hd.hybrid_decode_device_errors(wl.ctx):
            raise RuntimeError(f"device error flags in the {T}-token step")
        kvb = wl.token_pass_bytes()
        res.append({"tokens": T, "ms_per_step": round(ms, 4), "tokens_per_s": round(wl.B * T / (ms * 1e-3)),
                    "us_per_token": round(ms * 1e3 / T, 1), "speedup_vs_single_token_steps": round(T * single_ms / ms, 3),
                    "kv_bytes_read_per_step": kvb, "GBps": round(kvb / (ms * 1e-3) / 1e9, 1)})
        if (wl.Hq // wl.Hkv) * T == 16 and consumer == hd.HD_CONSUMER_TENSOR_CORE:
            # the same 16-row passes on tcgen05 (tensor memory), measured beside the default
            hd.hybrid_decode_set_consumer(wl.ctx, hd.HD_CONSUMER_TENSOR_MEMORY)
            ms_tm = time_steps(wl.step, args.steps, args.warmup, 1, device)
            if hd.hybrid_decode_device_errors(wl.ctx):
                raise RuntimeError(f"device error flags in the {T}-token step (tensor memory)")
            res[-1]["tensor_memory_consumer"] = {"ms_per_step": round(ms_tm, 4),
                                                 "GBps": round(kvb / (ms_tm * 1e-3) / 1e9, 1)}
        wl.ctx.close()
        del wl
        torch.cuda.empty_cache()
    return res


def roll_shift_bytes(wl) -> int:
    """Bytes a roll layout writes per step to shift its full windows down one
    row (K and V, every sliding layer), apart from the scored-key reads."""
    full = (wl.context >= synth.WINDOW).astype(np.int64) * (synth.WINDOW - 1)
    n_sliding = sum(1 for t in wl.types if t == synth.SLIDING)
    return int(full.sum()) * wl.Hkv * wl.row_bytes * n_sliding


def timed_workload(name, device, args, consumer, layout, read_peak) -> dict:
    """One workload's step (step grids on): ms per step, scored-KV GB/s, the grid
    alone by events, and fractions of the copy peak and of the read stream."""
    import torch
    import full_gqa_decode_gb300 as hd
    wl = Workload(name, device, seed=0, layout=layout)
    hd.hybrid_decode_set_consumer(wl.ctx, consumer)
    ms = time_steps(wl.step, args.steps, args.warmup, 1, device)
    hd.hybrid_decode_set_profiling(wl.ctx, hd.HD_PROFILE_STEP)
    for _ in range(3):
        wl.step()
    grid_ms, grid_n = hd.hybrid_decode_profile(wl.ctx, hd.HD_PROFILE_KIND_STEP)
    hd.hybrid_decode_set_profiling(wl.ctx, 0)
    hd.hybrid_decode_set_step_fusion(wl.ctx, False)
    per_layer_ms = time_steps(wl.step, args.steps, args.warmup, 1, device)
    hd.hybrid_decode_set_step_fusion(wl.ctx, True)
    flags = hd.hybrid_decode_device_errors(wl.ctx)
    if flags:
        raise RuntimeError(f"device error flags {flags:#x} in {name}")
    peak = measured_peaks()["hbm_gbs"]
    gbs = wl.bytes / (ms * 1e-3) / 1e9
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    plan = step_plan(wl.types, wl.B, wl.Hkv, wl.Hq // wl.Hkv, wl.max_ctx, wl.layout, "bf16", sms)
    res = {"ms_per_step": round(ms, 4), "us_per_step": round(ms * 1e3, 1), "value": round(gbs, 1), "unit": "GB/s",
           "kv_bytes_per_step": wl.bytes, "frac_of_peak_hbm": round(gbs / peak, 4),
           "frac_of_read_stream": round(gbs / read_peak, 4) if read_peak else None,
           "step_grid": dict(plan, chunks_per_full_sequence=-(-(wl.max_ctx + 1) // plan["chunk_keys"]))}
    if grid_n:
        avg = grid_ms / grid_n
        per_launch = wl.bytes * 3 // grid_n
        res["step_grid"].update({"launches_per_step": grid_n // 3, "avg_launch_ms": round(avg, 4),
                                 "achieved": round(per_launch / (avg * 1e-3) / 1e9, 1),
                                 "frac": round(per_launch / (avg * 1e-3) / 1e9 / peak, 4)})
    res["kernel_per_layer"] = {"ms_per_step": round(per_layer_ms, 4),
                               "value": round(wl.bytes / (per_layer_ms * 1e-3) / 1e9, 1), "unit": "GB/s"}
    if layout == synth.LAYOUT_ROLL:
        res["roll_shift_bytes_per_step"] = roll_shift_bytes(wl)
    wl.ctx.close()
    del wl
    torch.cuda.empty_cache()
    return res


def baseline_configs(device, args, consumer, read_peak) -> dict:
    """The other benchmark configurations, each as its own step: seven full layers
    at batch 4 and context 131072 (one chunk plan over the step grid), and the
    group-8 batch-256 mixed-length step with ring and with roll windows."""
    out = {"full7_b4_c131072": timed_workload("full7_b4_c131072", device, args, consumer, synth.LAYOUT_RING,
                                              read_peak)}
    g8 = {lay: timed_workload("step28_b256_g8_mixed", device, args, consumer,
                              synth.LAYOUT_RING if lay == "ring" else synth.LAYOUT_ROLL, read_peak)
          for lay in ("ring", "roll")}
    g8["roll_over_ring_time"] = round(g8["roll"]["ms_per_step"] / g8["ring"]["ms_per_step"], 4)
    g8["ring_saves"] = round(1.0 - g8["ring"]["ms_per_step"] / g8["roll"]["ms_per_step"], 4)
    out["step28_b256_g8_mixed"] = g8
    return out


def graph_steps(wl, args, device) -> float:
    """ms per step of the workload's step (in the context's current mode) captured
    once in a CUDA graph and replayed."""
    import torch
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        wl.step()
    torch.cuda.current_stream(device).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        wl.step()
    ms = time_steps(graph.replay, args.steps, args.warmup, 1, device)
    del graph
    return ms


def secondary_batch1(device, args, consumer) -> dict:
    """The 28-layer step at batch 1, context 4096 (launch-latency bound), launched
    eagerly and replayed from a CUDA graph of one decode_step."""
    import torch
    import full_gqa_decode_gb300 as hd
    wl = Workload(SECONDARY_WORKLOAD, device, seed=7)
    hd.hybrid_decode_set_consumer(wl.ctx, consumer)
    steps, warm = max(args.steps, 20), max(args.warmup, 3)
    ms = time_steps(wl.step, steps, warm, 1, device)
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        wl.step()
    torch.cuda.current_stream(device).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        wl.step()
    ms_graph = time_steps(graph.replay, steps, warm, 1, device)
    hd.hybrid_decode_set_step_fusion(wl.ctx, False)   # one kernel per layer, for comparison
    ms_layers = time_steps(wl.step, steps, warm, 1, device)
    hd.hybrid_decode_set_layer_overlap(wl.ctx, False)   # and every layer in full stream order
    ms_serial = time_steps(wl.step, steps, warm, 1, device)
    ms_serial_graph = graph_steps(wl, argparse.Namespace(steps=steps, warmup=warm), device)
    hd.hybrid_decode_set_layer_overlap(wl.ctx, True)
    hd.hybrid_decode_set_step_fusion(wl.ctx, True)
    if hd.hybrid_decode_device_errors(wl.ctx):
        raise RuntimeError("device error flags in the batch-1 step")
    return {"workload": SECONDARY_WORKLOAD, "us_per_step": round(ms * 1e3, 1),
            "us_per_step_cuda_graph": round(ms_graph * 1e3, 1),
            "us_per_step_kernel_per_layer": round(ms_layers * 1e3, 1),
            "us_per_step_layers_in_stream_order": round(ms_serial * 1e3, 1),
            "us_per_step_layers_in_stream_order_cuda_graph": round(ms_serial_graph * 1e3, 1),
            "kv_GBps_cuda_graph": round(wl.bytes / (ms_graph * 1e-3) / 1e9, 1),
            "kv_bytes_per_step": wl.bytes, "roofline_us": round(wl.bytes / (measured_peaks()["hbm_gbs"] * 1e9) * 1e6, 1)}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-secondary", dest="secondary", action="store_false")
    ap.add_argument("--consumer", choices=["tensor-core", "cuda-core", "tensor-memory"], default="tensor-core",
                    help="inner loop of the attention kernels (tensor-memory: tcgen05 for 16-row multi-token passes)")
    ap.add_argument("--layout", choices=["ring", "roll"], default="ring",
                    help="cache layout of the sliding layers")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="cache element type (fp8: E4M3 codes with per-kv-head scales)")
    ap.add_argument("--tokens", type=int, default=1, choices=range(1, 9), metavar="T",
                    help="new tokens per sequence and step (decode_step_tokens); GB/s then counts every pass's cache read")
    ap.add_argument("--fusion", choices=["on", "off"], default="on",
                    help="off: the timed steps run one kernel per layer (the dominant kernel is then the full layer's)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
