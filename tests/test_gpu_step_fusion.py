"""GPU parity of step grids (decode_step with step fusion, the default): the
attention of every layer of a step in one grid, with one chunk size planned
over all layers.  Outputs and lse against the oracle within the harness
tolerances, written caches bit-exact; launch counts show which path ran."""
import numpy as np
import pytest
import torch

import synth
from harness import FULL, RING, ROLL, SLIDING, LayerCase, assert_bits_equal, assert_lse_close, assert_out_close
from harness import oracle_layer

pytestmark = pytest.mark.gpu
D = synth.HEAD_DIM


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def launches(hd, ctx):
    return hd.hybrid_decode_launch_count(ctx)


class Step:
    """Seeded inputs of one decode_step over `types`, kept on the device."""

    def __init__(self, hd, rng, types, B, Hq, Hkv, context, layout, max_context, sink=None, kv="bf16"):
        self.types, self.layout = types, layout
        self.context = np.asarray(context, np.int32)
        self.cases, self.ios, self.dev = [], [], []
        for t in types:
            cap = (511 if layout == RING else 512) if t == SLIDING else max_context + 1
            case = LayerCase(rng, B, Hq, Hkv, cap, self.context, sink=sink, kv=kv)
            kd, vd = case.kc.cuda(), case.vc.cuda()
            out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
            lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
            keep = (case.q.cuda(), case.k.cuda(), case.v.cuda(), None if sink is None else sink.cuda())
            self.ios.append(hd.layer_io(keep[0], keep[1], keep[2], case.cache(hd, kd, vd, "cuda"), keep[3],
                                        out, lse))
            self.cases.append(case)
            self.dev.append((out, lse, kd, vd, keep))

    def run(self, hd, ctx, hint=0):
        hd.decode_step(ctx, torch.from_numpy(self.context).cuda(), self.ios, len(self.context), hint)
        torch.cuda.synchronize()
        assert hd.hybrid_decode_device_errors(ctx) == 0

    def check(self, orc):
        for i, (t, case) in enumerate(zip(self.types, self.cases)):
            ref = oracle_layer(orc, case, t, self.layout)
            out, lse, kd, vd, _ = self.dev[i]
            assert_out_close(out, ref["out"], f"layer {i} out")
            assert_lse_close(lse, ref["lse"], f"layer {i} lse")
            assert_bits_equal(kd, ref["kcache"], f"layer {i} K cache")
            assert_bits_equal(vd, ref["vcache"], f"layer {i} V cache")


def make_ctx(hd, types, B, max_context, layout=RING, Hq=8, Hkv=2, kv="bf16"):
    return hd.hybrid_decode_init(hd.Config(layer_types=types, num_q_heads=Hq, num_kv_heads=Hkv, max_batch=B,
                                           max_context=max_context, cache_layout=layout,
                                           kv_dtype=hd.HD_KV_FP8_E4M3 if kv == "fp8" else hd.HD_KV_BF16))


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_batch1_28_layer_step_is_one_grid(hd, orc, kv):
    """The batch-1 28-layer step at context 4096 (many short chunks, one CTA per
    SM): one launch, equal to the oracle layer by layer."""
    rng = synth.generator(1101)
    types = synth.SPARK_LAYER_TYPES
    ctx = make_ctx(hd, types, 1, 4096, kv=kv)
    step = Step(hd, rng, types, 1, 8, 2, [4096 - 1], RING, 4096, kv=kv)
    n0 = launches(hd, ctx)
    step.run(hd, ctx, hint=4096 - 1)
    assert launches(hd, ctx) - n0 == 1
    step.check(orc)
    ctx.close()


@pytest.mark.parametrize("fuse", [True, False])
@pytest.mark.parametrize("layout", [RING, ROLL])
def test_step_grid_launch_counts_and_parity(hd, orc, layout, fuse):
    """One grid for the 28 layers, roll windows included (the grid shifts them
    after reading); with fusion off, one kernel per layer (a roll layer's kernel
    shifts its own window after reading it)."""
    rng = synth.generator(1102)
    types = synth.SPARK_LAYER_TYPES
    ctx = make_ctx(hd, types, 4, 2048, layout=layout)
    hd.hybrid_decode_set_step_fusion(ctx, fuse)
    sink = synth.sink_vector(rng, ("normal", 1.0, 0.0), 8)
    step = Step(hd, rng, types, 4, 8, 2, [0, 511, 700, 2047], layout, 2048, sink=sink)
    n0 = launches(hd, ctx)
    step.run(hd, ctx)
    expect = 1 if fuse else len(types)
    assert launches(hd, ctx) - n0 == expect
    step.check(orc)
    ctx.close()


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_rolled_windows_shift_inside_the_grid_across_steps(hd, orc, kv):
    """Consecutive step grids over roll-layout layers from contexts that fill the
    512-row window: every step's outputs and the final windows match the oracle
    (the grid reads rows 1..511 of a full window, moves them down one row and
    stores the new entry at row 511)."""
    rng = synth.generator(1130)
    types = [SLIDING, FULL, SLIDING]
    B, Hq, Hkv, steps = 3, 8, 2, 6
    ctx = make_ctx(hd, types, B, 1200, layout=ROLL, kv=kv)
    start = np.array([508, 1, 900], np.int32)
    cases = [LayerCase(rng, B, Hq, Hkv, 512 if t == SLIDING else 1201, start, kv=kv) for t in types]
    host = [[synth.bits(c.kc), synth.bits(c.vc)] for c in cases]
    dev = [(c.kc.cuda(), c.vc.cuda()) for c in cases]
    for s_ in range(steps):
        context = start + s_
        ios, keep, refs = [], [], []
        for i, t in enumerate(types):
            q = synth.normal_bf16(rng, (B, Hq, D))
            k = synth.normal_bf16(rng, (B, Hkv, D))
            v = synth.normal_bf16(rng, (B, Hkv, D))
            rot, theta = synth.ROPE[t]
            c = cases[i]
            refs.append(orc.decode_layer(layer_type=t, layout=ROLL if t == SLIDING else 0, window=synth.WINDOW,
                                         rotary_dim=rot, rope_theta=theta, context=context, q=synth.bits(q),
                                         k=synth.bits(k), v=synth.bits(v), kcache=host[i][0], vcache=host[i][1],
                                         k_scale=None if c.k_scale is None else c.k_scale.numpy(),
                                         v_scale=None if c.v_scale is None else c.v_scale.numpy()))
            out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
            lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
            kk = (q.cuda(), k.cuda(), v.cuda(), out, lse)
            keep.append(kk)
            ios.append(hd.layer_io(kk[0], kk[1], kk[2], c.cache(hd, dev[i][0], dev[i][1], "cuda"), None, out, lse))
        n0 = launches(hd, ctx)
        hd.decode_step(ctx, torch.from_numpy(context).cuda(), ios, B)
        torch.cuda.synchronize()
        assert launches(hd, ctx) - n0 == 1
        assert hd.hybrid_decode_device_errors(ctx) == 0
        for i in range(len(types)):
            assert_out_close(keep[i][3], refs[i]["out"], f"step {s_} layer {i} out")
            assert_lse_close(keep[i][4], refs[i]["lse"], f"step {s_} layer {i} lse")
    for i in range(len(types)):
        assert_bits_equal(dev[i][0], host[i][0], f"layer {i} K cache")
        assert_bits_equal(dev[i][1], host[i][1], f"layer {i} V cache")
    ctx.close()


def test_more_layers_than_one_grid_holds(hd, orc):
    """40 layers: two grids (32 + 8 layers), same results."""
    rng = synth.generator(1103)
    types = [SLIDING, SLIDING, SLIDING, FULL] * 10
    ctx = make_ctx(hd, types, 2, 1500)
    step = Step(hd, rng, types, 2, 8, 2, [300, 1499], RING, 1500)
    n0 = launches(hd, ctx)
    step.run(hd, ctx)
    assert launches(hd, ctx) - n0 == 2
    step.check(orc)
    ctx.close()


@pytest.mark.parametrize("g", [1, 2, 8])
def test_step_grid_groups(hd, orc, g):
    rng = synth.generator(1110 + g)
    types = [SLIDING, FULL, SLIDING, FULL]
    Hkv = 2
    sink = synth.sink_vector(rng, ("normal", 2.0 ** 0.5, 0.25), g * Hkv)
    ctx = make_ctx(hd, types, 5, 3000, Hq=g * Hkv, Hkv=Hkv)
    step = Step(hd, rng, types, 5, g * Hkv, Hkv, [1, 510, 511, 1800, 2999], RING, 3000, sink=sink)
    step.run(hd, ctx)
    step.check(orc)
    ctx.close()


def test_aliased_outputs_run_layer_by_layer(hd, orc):
    """Layers that share one out/lse buffer are not independent: decode_step
    launches one kernel per layer in order, so the buffer ends with the last
    layer's result."""
    rng = synth.generator(1104)
    types = [SLIDING, FULL, SLIDING, FULL]
    B, Hq, Hkv = 2, 8, 2
    ctx = make_ctx(hd, types, B, 1024)
    step = Step(hd, rng, types, B, Hq, Hkv, [200, 900], RING, 1024)
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    for io in step.ios:
        io.out = out.data_ptr()
        io.lse = lse.data_ptr()
    n0 = launches(hd, ctx)
    step.run(hd, ctx)
    assert launches(hd, ctx) - n0 == len(types)
    ref = oracle_layer(orc, step.cases[-1], types[-1], RING)
    assert_out_close(out, ref["out"], "last layer out")
    assert_lse_close(lse, ref["lse"], "last layer lse")
    for i, (t, case) in enumerate(zip(types, step.cases)):
        r = oracle_layer(orc, case, t, RING)
        assert_bits_equal(step.dev[i][2], r["kcache"], f"layer {i} K cache")
        assert_bits_equal(step.dev[i][3], r["vcache"], f"layer {i} V cache")
    ctx.close()


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_fused_and_layer_by_layer_steps_agree(hd, kv):
    """The batch-16 block at contexts U[512, 32768] with and without step fusion:
    the same cache bits, outputs within the output tolerance of each other."""
    import bench
    dev = torch.device("cuda")
    runs, counts = [], []
    for fuse in (True, False):
        wl = bench.Workload("block4_b16_c512_32768", dev, seed=5, kv=kv)
        hd.hybrid_decode_set_step_fusion(wl.ctx, fuse)
        n0 = launches(hd, wl.ctx)
        wl.step()
        torch.cuda.synchronize()
        counts.append(launches(hd, wl.ctx) - n0)
        assert hd.hybrid_decode_device_errors(wl.ctx) == 0
        runs.append([(L["out"].float().cpu().double().numpy(), L["lse"].cpu().double().numpy(),
                      synth.bits(L["kc"]), synth.bits(L["vc"])) for L in wl.layers])
        wl.ctx.close()
    assert counts == [1, 4], counts
    for i, (a, b) in enumerate(zip(*runs)):
        assert np.array_equal(a[2], b[2]) and np.array_equal(a[3], b[3]), f"layer {i} caches differ"
        assert_out_close(torch.from_numpy(a[0]), b[0], f"layer {i} out")
        assert_lse_close(torch.from_numpy(a[1]), b[1], f"layer {i} lse")


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_lost_copy_in_a_step_grid_times_out_and_recovers(hd, orc, kv):
    """A copy that never arrives inside a step grid: the bounded waits run out
    (about one second), the grid reports HD_DEVERR_WAIT_TIMEOUT and returns; the
    same context then runs a correct step."""
    import time
    rng = synth.generator(1120)
    types = [SLIDING, FULL]
    ctx = make_ctx(hd, types, 2, 1024, kv=kv)
    bad = Step(hd, rng, types, 2, 8, 2, [300, 900], RING, 1024, kv=kv)
    hd.hybrid_decode_inject_lost_copy(ctx, 0)   # no stage arrives (chunks may be one stage long)
    n0 = launches(hd, ctx)
    t0 = time.time()
    hd.decode_step(ctx, torch.from_numpy(bad.context).cuda(), bad.ios, 2)
    flags = hd.hybrid_decode_device_errors(ctx)
    elapsed = time.time() - t0
    assert launches(hd, ctx) - n0 == 1
    assert flags & 8, f"expected a wait timeout, flags {flags:#x}"
    assert 0.5 < elapsed < 30.0, elapsed
    hd.hybrid_decode_inject_lost_copy(ctx, -1)
    good = Step(hd, rng, types, 2, 8, 2, [300, 900], RING, 1024, kv=kv)
    good.run(hd, ctx)
    good.check(orc)
    ctx.close()


@pytest.mark.parametrize("layout", [RING, ROLL])
def test_bad_contexts_in_a_step_grid_are_flagged_and_the_rest_served(hd, orc, layout):
    """Negative contexts and contexts past max_context inside one step grid: the
    device flags them, poisons those sequences' out/lse with NaN and leaves their
    caches alone; every other sequence of every layer is served correctly."""
    rng = synth.generator(1140)
    types = [SLIDING, FULL]
    B, Hq, Hkv = 4, 8, 2
    context = np.array([10, 150, -3, 60], np.int32)   # max_context 100
    ctx = make_ctx(hd, types, B, 100, layout=layout)
    cases = []
    for t in types:
        cap = (511 if layout == RING else 512) if t == SLIDING else 101
        c = LayerCase(rng, B, Hq, Hkv, cap, np.clip(context, 0, 100))
        c.context = context
        cases.append(c)
    ios, keep = [], []
    for c in cases:
        kk = (c.q.cuda(), c.k.cuda(), c.v.cuda(), c.kc.cuda(), c.vc.cuda(),
              torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda"),
              torch.empty(B, Hq, dtype=torch.float32, device="cuda"))
        keep.append(kk)
        ios.append(hd.layer_io(kk[0], kk[1], kk[2], hd.kv_cache(kk[3], kk[4]), None, kk[5], kk[6]))
    n0 = launches(hd, ctx)
    hd.decode_step(ctx, torch.from_numpy(context).cuda(), ios, B)
    torch.cuda.synchronize()
    assert launches(hd, ctx) - n0 == 1
    flags = hd.hybrid_decode_device_errors(ctx)
    assert flags & 1 and flags & 4, f"flags {flags:#x}"
    good, bad = [0, 3], [1, 2]
    for i, (t, c) in enumerate(zip(types, cases)):
        out, lse, kd, vd = keep[i][5], keep[i][6], keep[i][3], keep[i][4]
        assert torch.isnan(out[bad].float()).all() and torch.isnan(lse[bad]).all(), f"layer {i}"
        kc0, vc0 = synth.bits(c.kc), synth.bits(c.vc)
        assert np.array_equal(synth.bits(kd)[bad], kc0[bad]) and np.array_equal(synth.bits(vd)[bad], vc0[bad])
        sub = LayerCase(rng, 2, Hq, Hkv, c.kc.shape[2], context[good])
        sub.q, sub.k, sub.v = c.q[good], c.k[good], c.v[good]
        sub.kc, sub.vc = c.kc[good].contiguous(), c.vc[good].contiguous()
        ref = oracle_layer(orc, sub, t, layout)
        assert_out_close(out[good], ref["out"], f"layer {i} out")
        assert_lse_close(lse[good], ref["lse"], f"layer {i} lse")
        assert_bits_equal(kd[good], ref["kcache"], f"layer {i} K cache")
        assert_bits_equal(vd[good], ref["vcache"], f"layer {i} V cache")
    ctx.close()


def test_step_grid_replays_from_a_cuda_graph(hd, orc):
    """decode_step captured once in a CUDA graph and replayed over several steps:
    the grid's parameters (layer table, chunk plan) are fixed at capture, while the
    contexts, q/k/v and caches live in device buffers the replays update; every
    replay must equal the oracle's step."""
    rng = synth.generator(1150)
    types = [SLIDING, FULL, SLIDING, FULL]
    B, Hq, Hkv, hint = 2, 8, 2, 1200
    ctx = make_ctx(hd, types, B, hint)
    start = np.array([505, 40], np.int32)
    cases = [LayerCase(rng, B, Hq, Hkv, 511 if t == SLIDING else hint + 1, start) for t in types]
    host = [[synth.bits(c.kc), synth.bits(c.vc)] for c in cases]
    dev = [(c.kc.cuda(), c.vc.cuda()) for c in cases]
    ctx_d = torch.from_numpy(start).cuda()
    qkv = [(torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda"),
            torch.empty(B, Hkv, D, dtype=torch.bfloat16, device="cuda"),
            torch.empty(B, Hkv, D, dtype=torch.bfloat16, device="cuda")) for _ in types]
    outs = [(torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda"),
             torch.empty(B, Hq, dtype=torch.float32, device="cuda")) for _ in types]
    ios = hd.layer_array(ctx, [hd.layer_io(q, k, v, hd.kv_cache(*dev[i]), None, outs[i][0], outs[i][1])
                               for i, (q, k, v) in enumerate(qkv)])
    # one eager step on copies of the caches first (the kernel's one-time setup
    # happens outside the capture; the real caches stay as they are)
    spare = [(k.clone(), v.clone()) for k, v in dev]
    hd.decode_step(ctx, ctx_d, [hd.layer_io(q, k, v, hd.kv_cache(*spare[i]), None, outs[i][0], outs[i][1])
                                for i, (q, k, v) in enumerate(qkv)], B, hint)
    torch.cuda.synchronize()
    assert hd.hybrid_decode_device_errors(ctx) == 0
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):   # capture only: nothing runs, so the caches stay as they are
        with torch.cuda.graph(graph, stream=side):
            hd.decode_step(ctx, ctx_d, ios, B, hint, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for s_ in range(5):
        context = start + s_
        ctx_d.copy_(torch.from_numpy(context))
        refs = []
        for i, t in enumerate(types):
            q = synth.normal_bf16(rng, (B, Hq, D))
            k = synth.normal_bf16(rng, (B, Hkv, D))
            v = synth.normal_bf16(rng, (B, Hkv, D))
            for dst, src in zip(qkv[i], (q, k, v)):
                dst.copy_(src)
            rot, theta = synth.ROPE[t]
            refs.append(orc.decode_layer(layer_type=t, layout=RING if t == SLIDING else 0, window=synth.WINDOW,
                                         rotary_dim=rot, rope_theta=theta, context=context, q=synth.bits(q),
                                         k=synth.bits(k), v=synth.bits(v), kcache=host[i][0], vcache=host[i][1]))
        graph.replay()
        torch.cuda.synchronize()
        assert hd.hybrid_decode_device_errors(ctx) == 0
        for i in range(len(types)):
            assert_out_close(outs[i][0], refs[i]["out"], f"replay {s_} layer {i} out")
            assert_lse_close(outs[i][1], refs[i]["lse"], f"replay {s_} layer {i} lse")
    for i in range(len(types)):
        assert_bits_equal(dev[i][0], host[i][0], f"layer {i} K cache")
        assert_bits_equal(dev[i][1], host[i][1], f"layer {i} V cache")
    ctx.close()
