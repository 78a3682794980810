"""GPU parity: every call of the C ABI against the fp64 oracle on the same
seeded inputs (tolerances in harness.py; written cache entries bit-exact).

Caches are NaN beyond the entries a sequence has written, so reading a slot
the key set excludes shows up as a non-finite output."""
import numpy as np
import pytest
import torch

import synth
from harness import (FULL, RING, ROLL, SLIDING, LayerCase, assert_bits_equal, assert_lse_close,
                     assert_out_close, check_layer, gpu_layer, oracle_layer)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


CONSUMERS = ["tensor_core", "cuda_core"]


def make_ctx(hd, layer_types, Hq=8, Hkv=2, layout=0, max_batch=4, max_context=2048,
             consumer="tensor_core"):
    ctx = hd.hybrid_decode_init(hd.Config(layer_types=layer_types, num_q_heads=Hq, num_kv_heads=Hkv,
                                          cache_layout=layout, max_batch=max_batch,
                                          max_context=max_context))
    hd.hybrid_decode_set_consumer(ctx, hd.HD_CONSUMER_TENSOR_CORE if consumer == "tensor_core"
                                  else hd.HD_CONSUMER_CUDA_CORE)
    return ctx


def sink_for(rng, kind, Hq):
    if kind == "none":
        return None
    if kind == "normal":
        return synth.sink_vector(rng, ("normal", 1.0, 0.0), Hq)
    return synth.sink_vector(rng, ("normal", 2.0 ** 0.5, 0.25), Hq)  # a quarter at -inf


@pytest.mark.parametrize("consumer", CONSUMERS)
@pytest.mark.parametrize("c", [64, 700])
def test_tiny_hybrid_pair(hd, orc, c, consumer):
    """1 sliding (ring of 511) + 1 full layer, batch 2, 8/2 heads, sink N(0,1)."""
    rng = synth.generator(0)
    ctx = make_ctx(hd, [SLIDING, FULL], max_batch=2, max_context=1024, consumer=consumer)
    sink = synth.sink_vector(rng, ("normal", 1.0, 0.0), 8)
    check_layer(hd, orc, ctx, 0, SLIDING, RING, LayerCase(rng, 2, 8, 2, 511, [c, c], sink=sink))
    check_layer(hd, orc, ctx, 1, FULL, 0, LayerCase(rng, 2, 8, 2, 1025, [c, c], sink=sink))


RING_CONTEXTS = [0, 1, 31, 32, 33, 64, 200, 510, 511, 512, 513, 700, 1021, 1022, 1023, 5000]


@pytest.mark.parametrize("consumer", CONSUMERS)
@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("sink_kind", ["none", "normal", "neg_inf"])
def test_sliding_ring_contexts(hd, orc, g, sink_kind, consumer):
    rng = synth.generator(100 + g)
    B, Hkv = len(RING_CONTEXTS), 2
    ctx = make_ctx(hd, [SLIDING], Hq=g * Hkv, max_batch=B, max_context=5000, consumer=consumer)
    case = LayerCase(rng, B, g * Hkv, Hkv, 511, RING_CONTEXTS, sink=sink_for(rng, sink_kind, g * Hkv))
    check_layer(hd, orc, ctx, 0, SLIDING, RING, case)


FULL_CONTEXTS = [0, 1, 31, 32, 63, 64, 65, 127, 128, 511, 512, 513, 1000, 2047, 3001, 4096]


@pytest.mark.parametrize("consumer", CONSUMERS)
@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("sink_kind", ["none", "normal", "neg_inf"])
def test_full_contexts(hd, orc, g, sink_kind, consumer):
    rng = synth.generator(200 + g)
    B, Hkv = len(FULL_CONTEXTS), 2
    ctx = make_ctx(hd, [FULL], Hq=g * Hkv, max_batch=B, max_context=4096, consumer=consumer)
    case = LayerCase(rng, B, g * Hkv, Hkv, 4097, FULL_CONTEXTS, sink=sink_for(rng, sink_kind, g * Hkv))
    check_layer(hd, orc, ctx, 0, FULL, 0, case)


def test_full_context_hint_smaller_plan(hd, orc):
    """A call-specific context bound gives a finer split; results must not change."""
    rng = synth.generator(7)
    ctx = make_ctx(hd, [FULL], max_batch=3, max_context=8192)
    case = LayerCase(rng, 3, 8, 2, 8193, [100, 700, 1500], sink=sink_for(rng, "normal", 8))
    check_layer(hd, orc, ctx, 0, FULL, 0, case, max_context_hint=1500)


@pytest.mark.parametrize("g", [2, 4, 8])
def test_sliding_roll_contexts(hd, orc, g):
    rng = synth.generator(300 + g)
    contexts = [0, 1, 100, 510, 511, 512, 513, 600, 1024, 3000]
    B, Hkv = len(contexts), 2
    ctx = make_ctx(hd, [SLIDING], Hq=g * Hkv, layout=ROLL, max_batch=B, max_context=3000)
    case = LayerCase(rng, B, g * Hkv, Hkv, 512, contexts, sink=sink_for(rng, "neg_inf", g * Hkv))
    check_layer(hd, orc, ctx, 0, SLIDING, ROLL, case)


def test_sliding_equals_full_inside_window_on_gpu(hd):
    """With the full layer's RoPE on both, a sliding ring at c <= 510 scores the same keys."""
    rng = synth.generator(11)
    B, c = 2, 300
    ctx = hd.hybrid_decode_init(hd.Config(layer_types=[SLIDING, FULL], rotary_dim_sliding=64,
                                          rope_theta_sliding=5e6, max_batch=B, max_context=600))
    case = LayerCase(rng, B, 8, 2, 511, [c, c], sink=sink_for(rng, "normal", 8))
    full_k = torch.full((B, 2, 601, 256), float("nan"), dtype=torch.bfloat16)
    full_v = full_k.clone()
    full_k[:, :, :511] = case.kc
    full_v[:, :, :511] = case.vc
    a = gpu_layer(hd, ctx, 0, SLIDING, case)
    case.kc, case.vc = full_k, full_v
    b = gpu_layer(hd, ctx, 1, FULL, case)
    # Same keys, different split and order: equal to fp32 rounding.
    assert torch.allclose(a["out"].float(), b["out"].float(), atol=2e-2, rtol=2e-2)
    assert torch.allclose(a["lse"], b["lse"], atol=1e-4)


def test_multistep_lockstep(hd, orc):
    """150 consecutive decode steps of a ring, a roll and a full layer from contexts that
    cross the window; GPU caches and oracle caches must stay identical bit for bit."""
    rng = synth.generator(21)
    B, Hq, Hkv, D, steps = 2, 8, 2, 256, 150
    start = np.array([440, 505], np.int32)
    for layer_type, layout, cap in ((SLIDING, RING, 511), (SLIDING, ROLL, 512), (FULL, 0, 700)):
        ctx = make_ctx(hd, [layer_type], layout=layout, max_batch=B, max_context=699)
        case = LayerCase(rng, B, Hq, Hkv, cap, start, sink=sink_for(rng, "normal", Hq))
        kc_ref, vc_ref = synth.bits(case.kc), synth.bits(case.vc)
        kd, vd = case.kc.cuda(), case.vc.cuda()
        cache = hd.kv_cache(kd, vd)
        rot, theta = synth.ROPE[layer_type]
        for s in range(steps):
            context = start + s
            q = synth.normal_bf16(rng, (B, Hq, D))
            k = synth.normal_bf16(rng, (B, Hkv, D))
            v = synth.normal_bf16(rng, (B, Hkv, D))
            ref = orc.decode_layer(layer_type=layer_type, layout=layout, window=512, rotary_dim=rot,
                                   rope_theta=theta, context=context, q=synth.bits(q),
                                   k=synth.bits(k), v=synth.bits(v), kcache=kc_ref, vcache=vc_ref,
                                   sink=case.sink.numpy())
            ctx_d = torch.from_numpy(context).cuda()
            qrot = torch.empty(B, Hq, D, dtype=torch.float32, device="cuda")
            out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
            lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
            hd.rope_append_kv(ctx, 0, ctx_d, q.cuda(), k.cuda(), v.cuda(), qrot, cache)
            if layer_type == SLIDING:
                hd.decode_attn_sliding(ctx, 0, ctx_d, qrot, cache, case.sink.cuda(), out, lse)
            else:
                hd.decode_attn_full(ctx, 0, ctx_d, qrot, cache, case.sink.cuda(), out, lse)
            assert_out_close(out, ref["out"], f"out step {s}")
            assert_lse_close(lse, ref["lse"], f"lse step {s}")
        assert hd.hybrid_decode_device_errors(ctx) == 0
        assert_bits_equal(kd, kc_ref, f"K cache after {steps} steps ({layer_type}, {layout})")
        assert_bits_equal(vd, vc_ref, f"V cache after {steps} steps ({layer_type}, {layout})")


@pytest.mark.parametrize("consumer", CONSUMERS)
@pytest.mark.parametrize("layout", [RING, ROLL])
def test_decode_step_28_layers(hd, orc, layout, consumer):
    """decode_step over the 28-layer [S,S,S,F]x7 step vs the oracle layer by layer."""
    rng = synth.generator(31)
    B, Hq, Hkv, D = 2, 8, 2, 256
    context = np.array([700, 1500], np.int32)
    types = synth.SPARK_LAYER_TYPES
    ctx = make_ctx(hd, types, layout=layout, max_batch=B, max_context=2048, consumer=consumer)
    sink = synth.sink_vector(rng, ("normal", 1.0, 0.0), Hq)
    cases, ios, outs = [], [], []
    for t in types:
        cap = (511 if layout == RING else 512) if t == SLIDING else 2049
        case = LayerCase(rng, B, Hq, Hkv, cap, context, sink=sink)
        kd, vd = case.kc.cuda(), case.vc.cuda()
        out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
        dev_in = (case.q.cuda(), case.k.cuda(), case.v.cuda(), sink.cuda())
        ios.append(hd.layer_io(dev_in[0], dev_in[1], dev_in[2], hd.kv_cache(kd, vd), dev_in[3], out, lse))
        cases.append(case)
        outs.append((out, lse, kd, vd, dev_in))
    hd.decode_step(ctx, torch.from_numpy(context).cuda(), ios, B)
    torch.cuda.synchronize()
    assert hd.hybrid_decode_device_errors(ctx) == 0
    for i, (t, case) in enumerate(zip(types, cases)):
        ref = oracle_layer(orc, case, t, layout)
        out, lse, kd, vd, _ = outs[i]
        assert_out_close(out, ref["out"], f"layer {i} out")
        assert_lse_close(lse, ref["lse"], f"layer {i} lse")
        assert_bits_equal(kd, ref["kcache"], f"layer {i} K cache")
        assert_bits_equal(vd, ref["vcache"], f"layer {i} V cache")


@pytest.mark.parametrize("consumer", CONSUMERS)
def test_group8_mixed_lengths_with_neg_inf_sinks(hd, orc, consumer):
    """High-group shape: 16 q / 2 kv heads, 90% long and 10% short sequences,
    sink N(0, variance 2) with a quarter of the heads at -inf."""
    rng = synth.generator(41)
    B, Hq, Hkv = 20, 16, 2
    context = synth.context_lengths(rng, ("mixed", 2048, 0.10, 512), B)
    sink = synth.sink_vector(rng, ("normal", 2.0 ** 0.5, 0.25), Hq)
    ctx = make_ctx(hd, [SLIDING, FULL], Hq=Hq, max_batch=B, max_context=2048, consumer=consumer)
    check_layer(hd, orc, ctx, 0, SLIDING, RING, LayerCase(rng, B, Hq, Hkv, 511, context, sink=sink))
    check_layer(hd, orc, ctx, 1, FULL, 0, LayerCase(rng, B, Hq, Hkv, 2049, context, sink=sink))


@pytest.mark.parametrize("layout", [RING, ROLL])
def test_decode_step_multistep_lockstep(hd, orc, layout):
    """40 consecutive decode_step calls of a [S,S,S,F] block from contexts that cross
    the window; every output and, at the end, every cache equals the oracle's."""
    rng = synth.generator(51)
    B, Hq, Hkv, D, steps = 2, 8, 2, 256, 40
    types = [SLIDING, SLIDING, SLIDING, FULL]
    start = np.array([490, 3], np.int32)
    ctx = make_ctx(hd, types, layout=layout, max_batch=B, max_context=600)
    sink = synth.sink_vector(rng, ("normal", 1.0, 0.0), Hq)
    caps = [(511 if layout == RING else 512) if t == SLIDING else 601 for t in types]
    host = [[synth.bits(c) for c in (LayerCase(rng, B, Hq, Hkv, cap, start).kc,
                                      LayerCase(rng, B, Hq, Hkv, cap, start).vc)] for cap in caps]
    dev = [(synth.from_bits(k).cuda(), synth.from_bits(v).cuda()) for k, v in host]
    for s_ in range(steps):
        context = start + s_
        ios, outs, refs = [], [], []
        for i, t in enumerate(types):
            q = synth.normal_bf16(rng, (B, Hq, D))
            k = synth.normal_bf16(rng, (B, Hkv, D))
            v = synth.normal_bf16(rng, (B, Hkv, D))
            rot, theta = synth.ROPE[t]
            refs.append(orc.decode_layer(layer_type=t, layout=layout if t == SLIDING else 0, window=512,
                                         rotary_dim=rot, rope_theta=theta, context=context,
                                         q=synth.bits(q), k=synth.bits(k), v=synth.bits(v),
                                         kcache=host[i][0], vcache=host[i][1], sink=sink.numpy()))
            out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
            lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
            keep = (q.cuda(), k.cuda(), v.cuda(), sink.cuda())
            ios.append(hd.layer_io(keep[0], keep[1], keep[2], hd.kv_cache(*dev[i]), keep[3], out, lse))
            outs.append((out, lse, keep))
        hd.decode_step(ctx, torch.from_numpy(context).cuda(), ios, B)
        for i in range(len(types)):
            assert_out_close(outs[i][0], refs[i]["out"], f"step {s_} layer {i} out")
            assert_lse_close(outs[i][1], refs[i]["lse"], f"step {s_} layer {i} lse")
    assert hd.hybrid_decode_device_errors(ctx) == 0
    for i in range(len(types)):
        assert_bits_equal(dev[i][0], host[i][0], f"layer {i} K cache")
        assert_bits_equal(dev[i][1], host[i][1], f"layer {i} V cache")


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_layer_overlap_changes_no_bit(hd, kv):
    """decode_step layer by layer (no step fusion) with and without the layer
    overlap (a layer starting before the previous one finishes) computes the same
    bits: outputs, lse and caches."""
    import bench
    dev = torch.device("cuda")
    runs = []
    for overlap in (True, False):
        wl = bench.Workload("block4_b16_c512_32768", dev, seed=3, kv=kv)
        hd.hybrid_decode_set_step_fusion(wl.ctx, False)
        hd.hybrid_decode_set_layer_overlap(wl.ctx, overlap)
        wl.step()
        torch.cuda.synchronize()
        assert hd.hybrid_decode_device_errors(wl.ctx) == 0
        runs.append([(synth.bits(L["out"]), L["lse"].cpu().numpy(), synth.bits(L["kc"]), synth.bits(L["vc"]))
                     for L in wl.layers])
        wl.ctx.close()
    for i, (a, b) in enumerate(zip(*runs)):
        for x, y in zip(a, b):
            assert np.array_equal(x, y), f"layer {i} differs with the overlap"


@pytest.mark.parametrize("cluster", [True, False])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_single_layer_chunk_merge_paths(hd, orc, g, cluster):
    """Single-layer calls on small grids merge their chunks inside a thread-block
    cluster (up to 16 chunks per (sequence, kv head), the default) or through the
    workspace: both against the oracle, for a full layer whose longest sequence
    needs more chunks than a cluster holds and a sliding ring layer."""
    rng = synth.generator(1500 + g)
    B, Hkv = 3, 2
    contexts = [0, 1500, 6000]
    ctx = make_ctx(hd, [SLIDING, FULL], Hq=g * Hkv, max_batch=B, max_context=6000)
    hd.hybrid_decode_set_cluster_combine(ctx, cluster)
    sink = sink_for(rng, "neg_inf", g * Hkv)
    check_layer(hd, orc, ctx, 0, SLIDING, RING, LayerCase(rng, B, g * Hkv, Hkv, 511, contexts, sink=sink))
    check_layer(hd, orc, ctx, 1, FULL, 0, LayerCase(rng, B, g * Hkv, Hkv, 6001, contexts, sink=sink))
    # the same layers again: the merge leaves nothing behind that the next call reads
    check_layer(hd, orc, ctx, 1, FULL, 0, LayerCase(rng, B, g * Hkv, Hkv, 6001, [6000, 3, 2047], sink=sink))
    ctx.close()


def _near_midpoint_keys(orc, rng, context, Hkv, layer_type, tries=20000):
    """New keys [B][Hkv][256] (bf16 bits) whose rotated pairs land within three
    binary32 units of a bf16 rounding midpoint: the first output of even pairs,
    the second of odd pairs.  Such values take the kernels' binary64 rounding
    path; found by seeded random search (the expected bits come from the oracle)."""
    rot, theta = synth.ROPE[layer_type]
    half = rot // 2
    B = len(context)
    keys = synth.bits(synth.normal_bf16(rng, (B, Hkv, synth.HEAD_DIM)))
    even = (np.arange(half) % 2 == 0)[:, None]
    for b in range(B):
        cs, sn = orc.rope_angles(int(context[b]), rot, theta)
        c, s = cs.astype(np.float64)[:, None], sn.astype(np.float64)[:, None]
        for h in range(Hkv):
            f = rng.standard_normal((2, half, tries)).astype(np.float32).view(np.uint32)
            cand = ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)       # nearest-even bf16
            x1 = (cand[0].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            x2 = (cand[1].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            y = np.where(even, x1 * c - x2 * s, x2 * c + x1 * s)                # exact products, one rounding
            low = (y.astype(np.float32).view(np.uint32) & 0xFFFF).astype(np.int64)
            ok = (np.abs(low - 0x8000) <= 3) & (y != 0)
            for i in range(half):
                hit = np.flatnonzero(ok[i])
                if len(hit):
                    keys[b, h, i], keys[b, h, i + half] = cand[0, i, hit[0]], cand[1, i, hit[0]]
    return keys


@pytest.mark.parametrize("layer_type", [SLIDING, FULL])
def test_new_keys_near_bf16_rounding_midpoints(hd, orc, layer_type):
    """The written key is bf16_rne(x1 c - x2 s) of the exact rotation.  Keys whose
    rotation sits next to a bf16 rounding midpoint -- where the kernels' binary32
    evaluation defers to binary64 -- are stored bit-exactly, both by decode_step
    (rotated in the attention kernel) and by rope_append_kv."""
    rng = synth.generator(1600 + layer_type)
    B, Hq, Hkv = 3, 8, 2
    context = np.array([5, 700, 3000], np.int32)
    cap = 511 if layer_type == SLIDING else 3001
    case = LayerCase(rng, B, Hq, Hkv, cap, context)
    case.k = torch.from_numpy(_near_midpoint_keys(orc, rng, context, Hkv, layer_type).view(np.int16)).view(torch.bfloat16)
    ref = oracle_layer(orc, case, layer_type, RING)
    # decode_step: the attention kernel rotates and stores the entry
    ctx = make_ctx(hd, [layer_type], max_batch=B, max_context=3000)
    kd, vd = case.kc.cuda(), case.vc.cuda()
    out = torch.empty(B, Hq, 256, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    dev = (case.q.cuda(), case.k.cuda(), case.v.cuda())
    io = [hd.layer_io(dev[0], dev[1], dev[2], hd.kv_cache(kd, vd), None, out, lse)]
    hd.decode_step(ctx, torch.from_numpy(context).cuda(), io, B)
    torch.cuda.synchronize()
    assert hd.hybrid_decode_device_errors(ctx) == 0
    assert_bits_equal(kd, ref["kcache"], "K cache written by decode_step")
    assert_out_close(out, ref["out"])
    # rope_append_kv + the attention call: the rope kernel stores the entry
    ctx2 = make_ctx(hd, [layer_type], max_batch=B, max_context=3000)
    got = check_layer(hd, orc, ctx2, 0, layer_type, RING, case)
    ctx.close()
    ctx2.close()
