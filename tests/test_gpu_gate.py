"""GPU parity of the optional per-head sigmoid output gate, fused into the
attention epilogue (spark_export.py, `_Layer.forward`: each head's attention
output times sigmoid of its gate logit).  Every gated case is checked against
the oracle with the harness tolerances; lse must not depend on the gate."""
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


def make_ctx(hd, layer_types, Hq=8, Hkv=2, layout=0, max_batch=4, max_context=2048,
             consumer=None):
    ctx = hd.hybrid_decode_init(hd.Config(layer_types=layer_types, num_q_heads=Hq, num_kv_heads=Hkv,
                                          cache_layout=layout, max_batch=max_batch,
                                          max_context=max_context))
    if consumer is not None:
        hd.hybrid_decode_set_consumer(ctx, consumer)
    return ctx


CONSUMERS = ["tensor_core", "cuda_core"]


def _consumer(hd, name):
    return hd.HD_CONSUMER_TENSOR_CORE if name == "tensor_core" else hd.HD_CONSUMER_CUDA_CORE


@pytest.mark.parametrize("consumer", CONSUMERS)
@pytest.mark.parametrize("g", [1, 8])
def test_gated_ring_and_full(hd, orc, g, consumer):
    """Ring and full layers over contexts that take one chunk and many, with a sink
    and gate logits that include +inf, -inf, 0 and +-30 for the first sequence."""
    rng = synth.generator(500 + g)
    contexts = [700, 0, 33, 510, 511, 1500, 3001]
    B, Hkv = len(contexts), 2
    Hq = g * Hkv
    ctx = make_ctx(hd, [SLIDING, FULL], Hq=Hq, max_batch=B, max_context=3001,
                   consumer=_consumer(hd, consumer))
    sink = synth.sink_vector(rng, ("normal", 1.0, 0.0), Hq)
    for layer, t, cap in ((0, SLIDING, 511), (1, FULL, 3002)):
        case = LayerCase(rng, B, Hq, Hkv, cap, contexts, sink=sink,
                         gate=synth.gate_logits(rng, B, Hq, std=2.0, specials=True))
        ref, got = check_layer(hd, orc, ctx, layer, t, RING, case)
        # +inf passes the head through, -inf zeroes it (head cycle of the specials)
        heads = np.arange(Hq)
        assert torch.all(got["out"][0, heads[heads % 5 == 1]].float() == 0)


def test_gated_roll(hd, orc):
    rng = synth.generator(511)
    contexts = [0, 100, 511, 512, 1024]
    B, Hq, Hkv = len(contexts), 8, 2
    ctx = make_ctx(hd, [SLIDING], layout=ROLL, max_batch=B, max_context=1024)
    case = LayerCase(rng, B, Hq, Hkv, 512, contexts, sink=synth.sink_vector(rng, ("normal", 1.0, 0.25), Hq),
                     gate=synth.gate_logits(rng, B, Hq, std=2.0, specials=True))
    check_layer(hd, orc, ctx, 0, SLIDING, ROLL, case)


def test_gate_leaves_lse_and_scales_out(hd):
    """Gated and ungated runs on the same inputs: lse identical bit for bit and
    out equal to the ungated out times sigmoid(logit), within bf16 rounding."""
    rng = synth.generator(512)
    B, Hq, Hkv = 3, 8, 2
    ctx = make_ctx(hd, [FULL], max_batch=B, max_context=4096)
    case = LayerCase(rng, B, Hq, Hkv, 4097, [4000, 900, 64], sink=synth.sink_vector(rng, ("normal", 1.0, 0.0), Hq))
    plain = gpu_layer(hd, ctx, 0, FULL, case)
    case.gate = synth.gate_logits(rng, B, Hq, std=3.0)
    gated = gpu_layer(hd, ctx, 0, FULL, case)
    assert plain["flags"] == 0 and gated["flags"] == 0
    assert torch.equal(plain["lse"], gated["lse"])
    factor = torch.sigmoid(case.gate.double()).cuda()[:, :, None]
    want = plain["out"].double() * factor
    err = (gated["out"].double() - want).abs()
    assert torch.all(err <= 2 * 2.0 ** -8 * want.abs() + 1e-6)


def test_gate_long_context_many_chunks(hd, orc):
    """Full layer at context 65536 (split into many chunks): the gate is applied once,
    in the cross-chunk combine."""
    rng = synth.generator(513)
    B, Hq, Hkv, c = 2, 8, 2, 65536
    ctx = make_ctx(hd, [FULL], max_batch=B, max_context=c)
    ck, nc = hd.hd_plan_split(B, Hkv, c + 1, torch.cuda.get_device_properties(0).multi_processor_count)
    assert nc > 1
    case = LayerCase(rng, B, Hq, Hkv, c + 1, [c, c - 777], sink=synth.sink_vector(rng, ("normal", 1.0, 0.0), Hq),
                     gate=synth.gate_logits(rng, B, Hq, std=2.0))
    check_layer(hd, orc, ctx, 0, FULL, 0, case)


@pytest.mark.parametrize("layout", [RING, ROLL])
def test_gated_decode_step(hd, orc, layout):
    """decode_step over [S,S,S,F] x 2 with per-layer gate logits (and no gate on one
    layer) vs the oracle layer by layer, caches bit-exact."""
    rng = synth.generator(514)
    B, Hq, Hkv, D = 3, 8, 2, 256
    context = np.array([700, 1500, 5], np.int32)
    types = [SLIDING, SLIDING, SLIDING, FULL] * 2
    ctx = make_ctx(hd, types, layout=layout, max_batch=B, max_context=2048)
    sink = synth.sink_vector(rng, ("normal", 1.0, 0.0), Hq)
    cases, ios, keep = [], [], []
    for i, t in enumerate(types):
        cap = (511 if layout == RING else 512) if t == SLIDING else 2049
        gate = None if i == 2 else synth.gate_logits(rng, B, Hq, std=2.0, specials=(i == 3))
        case = LayerCase(rng, B, Hq, Hkv, cap, context, sink=sink, gate=gate)
        kd, vd = case.kc.cuda(), case.vc.cuda()
        out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
        dev_in = (case.q.cuda(), case.k.cuda(), case.v.cuda(), sink.cuda(),
                  None if gate is None else gate.cuda())
        ios.append(hd.layer_io(dev_in[0], dev_in[1], dev_in[2], hd.kv_cache(kd, vd), dev_in[3], out, lse,
                               gate=dev_in[4]))
        cases.append(case)
        keep.append((out, lse, kd, vd, dev_in))
    hd.decode_step(ctx, torch.from_numpy(context).cuda(), ios, B)
    torch.cuda.synchronize()
    assert hd.hybrid_decode_device_errors(ctx) == 0
    for i, (t, case) in enumerate(zip(types, cases)):
        ref = oracle_layer(orc, case, t, layout)
        out, lse, kd, vd, _ = keep[i]
        assert_out_close(out, ref["out"], f"layer {i} out")
        assert_lse_close(lse, ref["lse"], f"layer {i} lse")
        assert_bits_equal(kd, ref["kcache"], f"layer {i} K cache")
        assert_bits_equal(vd, ref["vcache"], f"layer {i} V cache")


def test_gate_shape_is_checked(hd):
    rng = synth.generator(515)
    ctx = make_ctx(hd, [FULL], max_batch=2, max_context=128)
    case = LayerCase(rng, 2, 8, 2, 129, [10, 20], gate=torch.zeros(2, 4))
    with pytest.raises(ValueError):
        gpu_layer(hd, ctx, 0, FULL, case)
    case.gate = torch.zeros(2, 8, dtype=torch.float64)
    with pytest.raises(ValueError):
        gpu_layer(hd, ctx, 0, FULL, case)
