"""GPU parity of the FP8 (E4M3) KV cache with per-kv-head K and V scales
against the oracle on the same codes: every written code bit-exact, outputs
within the harness tolerances.  Unwritten entries hold the NaN code, so a read
of an excluded slot shows up as a non-finite output."""
import numpy as np
import pytest
import torch

import synth
from harness import (FULL, RING, ROLL, SLIDING, LayerCase, assert_bits_equal, assert_lse_close,
                     assert_out_close, check_layer, oracle_layer)

pytestmark = pytest.mark.gpu

CONSUMERS = ["tensor_core", "cuda_core"]
RING_CONTEXTS = [0, 1, 31, 32, 33, 64, 200, 510, 511, 512, 513, 700, 1021, 1022, 1023, 5000]
FULL_CONTEXTS = [0, 1, 31, 32, 63, 64, 65, 127, 128, 511, 512, 513, 1000, 2047, 3001, 4096]


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def make_ctx(hd, layer_types, Hq=8, Hkv=2, layout=0, max_batch=4, max_context=2048, consumer="tensor_core"):
    ctx = hd.hybrid_decode_init(hd.Config(layer_types=layer_types, num_q_heads=Hq, num_kv_heads=Hkv,
                                          cache_layout=layout, max_batch=max_batch, max_context=max_context,
                                          kv_dtype=hd.HD_KV_FP8_E4M3))
    hd.hybrid_decode_set_consumer(ctx, hd.HD_CONSUMER_TENSOR_CORE if consumer == "tensor_core"
                                  else hd.HD_CONSUMER_CUDA_CORE)
    return ctx


def sink_for(rng, kind, Hq):
    if kind == "none":
        return None
    if kind == "normal":
        return synth.sink_vector(rng, ("normal", 1.0, 0.0), Hq)
    return synth.sink_vector(rng, ("normal", 2.0 ** 0.5, 0.25), Hq)


@pytest.mark.parametrize("consumer", CONSUMERS)
@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("sink_kind", ["none", "neg_inf"])
def test_fp8_ring_contexts(hd, orc, g, sink_kind, consumer):
    rng = synth.generator(600 + g)
    B, Hkv = len(RING_CONTEXTS), 2
    ctx = make_ctx(hd, [SLIDING], Hq=g * Hkv, max_batch=B, max_context=5000, consumer=consumer)
    case = LayerCase(rng, B, g * Hkv, Hkv, 511, RING_CONTEXTS, sink=sink_for(rng, sink_kind, g * Hkv), kv="fp8")
    check_layer(hd, orc, ctx, 0, SLIDING, RING, case)


@pytest.mark.parametrize("consumer", CONSUMERS)
@pytest.mark.parametrize("g", [1, 4, 8])
def test_fp8_full_contexts(hd, orc, g, consumer):
    rng = synth.generator(610 + g)
    B, Hkv = len(FULL_CONTEXTS), 2
    ctx = make_ctx(hd, [FULL], Hq=g * Hkv, max_batch=B, max_context=4096, consumer=consumer)
    case = LayerCase(rng, B, g * Hkv, Hkv, 4097, FULL_CONTEXTS, sink=sink_for(rng, "normal", g * Hkv), kv="fp8")
    check_layer(hd, orc, ctx, 0, FULL, 0, case)


@pytest.mark.parametrize("g", [2, 8])
def test_fp8_roll_contexts(hd, orc, g):
    rng = synth.generator(620 + g)
    contexts = [0, 1, 100, 510, 511, 512, 513, 600, 1024, 3000]
    B, Hkv = len(contexts), 2
    ctx = make_ctx(hd, [SLIDING], Hq=g * Hkv, layout=ROLL, max_batch=B, max_context=3000)
    case = LayerCase(rng, B, g * Hkv, Hkv, 512, contexts, sink=sink_for(rng, "neg_inf", g * Hkv), kv="fp8")
    check_layer(hd, orc, ctx, 0, SLIDING, ROLL, case)


def test_fp8_saturating_new_entries(hd, orc):
    """New keys and values far beyond 448 * scale: the written codes saturate to +-448
    exactly as the oracle's, on the ring, full and roll paths."""
    rng = synth.generator(630)
    for layer_type, layout, cap in ((SLIDING, RING, 511), (FULL, 0, 1025), (SLIDING, ROLL, 512)):
        ctx = make_ctx(hd, [layer_type], layout=layout if layer_type == SLIDING else 0, max_batch=3,
                       max_context=1024)
        case = LayerCase(rng, 3, 8, 2, cap, [5, 600, 1024], kv="fp8", k_std=40.0,
                         sink=sink_for(rng, "normal", 8))
        ref, got = check_layer(hd, orc, ctx, 0, layer_type, layout, case)
        assert np.any((synth.bits(got["kcache"]) & 0x7F) == 0x7E), "no saturated code was written"


def test_fp8_long_context_many_chunks(hd, orc):
    rng = synth.generator(640)
    B, Hq, Hkv, c = 2, 8, 2, 65536
    ctx = make_ctx(hd, [FULL], max_batch=B, max_context=c)
    case = LayerCase(rng, B, Hq, Hkv, c + 1, [c, c - 999], sink=sink_for(rng, "normal", Hq), kv="fp8",
                     gate=synth.gate_logits(rng, B, Hq, std=2.0))
    check_layer(hd, orc, ctx, 0, FULL, 0, case)


@pytest.mark.parametrize("consumer", CONSUMERS)
@pytest.mark.parametrize("layout", [RING, ROLL])
def test_fp8_decode_step_28_layers(hd, orc, layout, consumer):
    """decode_step over the 28-layer step with E4M3 caches: the new entry is rotated,
    quantised, scored and stored inside the layer kernel."""
    rng = synth.generator(650)
    B, Hq, Hkv, D = 2, 8, 2, 256
    context = np.array([700, 1500], np.int32)
    types = synth.SPARK_LAYER_TYPES
    ctx = make_ctx(hd, types, layout=layout, max_batch=B, max_context=2048, consumer=consumer)
    sink = synth.sink_vector(rng, ("normal", 1.0, 0.0), Hq)
    cases, ios, keep = [], [], []
    for t in types:
        cap = (511 if layout == RING else 512) if t == SLIDING else 2049
        case = LayerCase(rng, B, Hq, Hkv, cap, context, sink=sink, kv="fp8")
        kd, vd = case.kc.cuda(), case.vc.cuda()
        out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
        dev_in = (case.q.cuda(), case.k.cuda(), case.v.cuda(), sink.cuda())
        cache = case.cache(hd, kd, vd, torch.device("cuda"))
        ios.append(hd.layer_io(dev_in[0], dev_in[1], dev_in[2], cache, dev_in[3], out, lse))
        cases.append(case)
        keep.append((out, lse, kd, vd, dev_in, cache))
    hd.decode_step(ctx, torch.from_numpy(context).cuda(), ios, B)
    torch.cuda.synchronize()
    assert hd.hybrid_decode_device_errors(ctx) == 0
    for i, (t, case) in enumerate(zip(types, cases)):
        ref = oracle_layer(orc, case, t, layout)
        out, lse, kd, vd = keep[i][:4]
        assert_out_close(out, ref["out"], f"layer {i} out")
        assert_lse_close(lse, ref["lse"], f"layer {i} lse")
        assert_bits_equal(kd, ref["kcache"], f"layer {i} K codes")
        assert_bits_equal(vd, ref["vcache"], f"layer {i} V codes")


@pytest.mark.parametrize("layout", [RING, ROLL])
def test_fp8_step_grid_three_ctas_per_sm(hd, orc, layout):
    """A group-4 E4M3 step grid with more CTAs than SMs (three CTAs per SM on
    two-stage rings): full layers in several chunks with a ragged last one, sliding
    layers in one, contexts from empty to the bound; every layer against the oracle."""
    import math
    rng = synth.generator(655)
    B, Hq, Hkv, D, mc = 8, 8, 2, 256, 3000
    context = np.array([0, 1, 511, 512, 1024, 1500, 2047, mc - 1], np.int32)
    types = synth.SPARK_LAYER_TYPES
    keys = [511 if t == SLIDING else mc + 1 for t in types]
    chunk = hd.hd_plan_step_split(keys, B, Hkv, Hq // Hkv, 152, kv_dtype=hd.HD_KV_FP8_E4M3)
    ctas = sum(B * Hkv * max(1, math.ceil(k / chunk)) for k in keys)
    assert ctas > torch.cuda.get_device_properties(0).multi_processor_count
    ctx = make_ctx(hd, types, layout=layout, max_batch=B, max_context=mc)
    sink = synth.sink_vector(rng, ("normal", 2.0 ** 0.5, 0.25), Hq)
    cases, ios, keep = [], [], []
    for t in types:
        cap = (511 if layout == RING else 512) if t == SLIDING else mc + 1
        case = LayerCase(rng, B, Hq, Hkv, cap, context, sink=sink, kv="fp8")
        kd, vd = case.kc.cuda(), case.vc.cuda()
        out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
        dev_in = (case.q.cuda(), case.k.cuda(), case.v.cuda(), sink.cuda())
        cache = case.cache(hd, kd, vd, torch.device("cuda"))
        ios.append(hd.layer_io(dev_in[0], dev_in[1], dev_in[2], cache, dev_in[3], out, lse))
        cases.append(case)
        keep.append((out, lse, kd, vd, dev_in, cache))
    launches = hd.hybrid_decode_launch_count(ctx)
    hd.decode_step(ctx, torch.from_numpy(context).cuda(), ios, B)
    torch.cuda.synchronize()
    assert hd.hybrid_decode_launch_count(ctx) - launches == 1, "one step grid"
    assert hd.hybrid_decode_device_errors(ctx) == 0
    for i, (t, case) in enumerate(zip(types, cases)):
        ref = oracle_layer(orc, case, t, layout)
        out, lse, kd, vd = keep[i][:4]
        assert_out_close(out, ref["out"], f"layer {i} out")
        assert_lse_close(lse, ref["lse"], f"layer {i} lse")
        assert_bits_equal(kd, ref["kcache"], f"layer {i} K codes")
        assert_bits_equal(vd, ref["vcache"], f"layer {i} V codes")


@pytest.mark.parametrize("layout", [RING, ROLL])
def test_fp8_decode_step_multistep_lockstep(hd, orc, layout):
    """30 consecutive decode_step calls of a [S,S,S,F] block across the window: every
    output and, at the end, every cache code equals the oracle's."""
    rng = synth.generator(660)
    B, Hq, Hkv, D, steps = 2, 8, 2, 256, 30
    types = [SLIDING, SLIDING, SLIDING, FULL]
    start = np.array([495, 3], np.int32)
    ctx = make_ctx(hd, types, layout=layout, max_batch=B, max_context=600)
    sink = synth.sink_vector(rng, ("normal", 1.0, 0.0), Hq)
    caps = [(511 if layout == RING else 512) if t == SLIDING else 601 for t in types]
    proto = [LayerCase(rng, B, Hq, Hkv, cap, start, kv="fp8") for cap in caps]
    host = [[synth.bits(p.kc), synth.bits(p.vc)] for p in proto]
    dev = [(p.kc.cuda(), p.vc.cuda()) for p in proto]
    caches = [p.cache(hd, *dev[i], torch.device("cuda")) for i, p in enumerate(proto)]
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
                                         kcache=host[i][0], vcache=host[i][1], sink=sink.numpy(),
                                         k_scale=proto[i].k_scale.numpy(), v_scale=proto[i].v_scale.numpy()))
            out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
            lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
            keep = (q.cuda(), k.cuda(), v.cuda(), sink.cuda())
            ios.append(hd.layer_io(keep[0], keep[1], keep[2], caches[i], keep[3], out, lse))
            outs.append((out, lse, keep))
        hd.decode_step(ctx, torch.from_numpy(context).cuda(), ios, B)
        for i in range(len(types)):
            assert_out_close(outs[i][0], refs[i]["out"], f"step {s_} layer {i} out")
            assert_lse_close(outs[i][1], refs[i]["lse"], f"step {s_} layer {i} lse")
    assert hd.hybrid_decode_device_errors(ctx) == 0
    for i in range(len(types)):
        assert_bits_equal(dev[i][0], host[i][0], f"layer {i} K codes")
        assert_bits_equal(dev[i][1], host[i][1], f"layer {i} V codes")


def test_fp8_cache_needs_fp8_context(hd):
    """Scales on a bf16 context, or a bf16 cache on an FP8 context, are argument errors."""
    rng = synth.generator(670)
    case = LayerCase(rng, 2, 8, 2, 129, [10, 20], kv="fp8")
    bf16_ctx = hd.hybrid_decode_init(hd.Config(layer_types=[FULL], max_batch=2, max_context=128))
    fp8_ctx = make_ctx(hd, [FULL], max_batch=2, max_context=128)
    dev = torch.device("cuda")
    qrot = torch.zeros(2, 8, 256, device=dev)
    out = torch.empty(2, 8, 256, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(2, 8, device=dev)
    ctx_d = torch.from_numpy(case.context).to(dev)
    fp8_cache = case.cache(hd, case.kc.to(dev), case.vc.to(dev), dev)
    bf16_cache = hd.kv_cache(torch.zeros(2, 2, 129, 256, dtype=torch.bfloat16, device=dev),
                             torch.zeros(2, 2, 129, 256, dtype=torch.bfloat16, device=dev))
    with pytest.raises(hd.HDError) as e:
        hd.decode_attn_full(bf16_ctx, 0, ctx_d, qrot, fp8_cache, None, out, lse)
    assert e.value.status == 1
    with pytest.raises(hd.HDError) as e:
        hd.decode_attn_full(fp8_ctx, 0, ctx_d, qrot, bf16_cache, None, out, lse)
    assert e.value.status == 1
    bf16_ctx.close()
    fp8_ctx.close()


def test_fp8_quantisation_at_midpoints(hd, orc):
    """New keys and values placed exactly on E4M3 rounding midpoints (times a
    power-of-two scale, so the quotient is exact) and one bf16 step either side
    of them: every written code must equal the oracle's (ties to even)."""
    torch_codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    vals = torch_codes.view(torch.float8_e4m3fn).float().numpy()
    pos = np.unique(vals[np.isfinite(vals) & (vals >= 0)])
    mids = (pos[:-1] + pos[1:]) / 2
    mids = np.concatenate([mids, mids * (1 + 2.0 ** -7), mids * (1 - 2.0 ** -8), -mids])  # bf16 neighbours, signs
    scale = 2.0 ** -5
    B, Hq, Hkv = 4, 8, 2
    n = B * Hkv * synth.HEAD_DIM
    x = np.resize(mids * scale, n).astype(np.float32).reshape(B, Hkv, synth.HEAD_DIM)
    rng = synth.generator(680)
    ctx = make_ctx(hd, [FULL], max_batch=B, max_context=64)
    case = LayerCase(rng, B, Hq, Hkv, 65, [0] * B, kv="fp8")   # position 0: the key is not rotated
    case.k = torch.from_numpy(x).to(torch.bfloat16)
    case.v = torch.from_numpy(x[::-1].copy()).to(torch.bfloat16)
    case.k_scale = torch.full((Hkv,), scale, dtype=torch.float32)
    case.v_scale = torch.full((Hkv,), scale, dtype=torch.float32)
    check_layer(hd, orc, ctx, 0, FULL, 0, case)
