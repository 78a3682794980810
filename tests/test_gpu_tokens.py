"""GPU parity of multi-token decode (decode_step_tokens): T new tokens per
sequence, each attending causally to its window, against the oracle's
multi-token step (T single-token steps in order).  Written cache entries are
bit-exact; outputs and lse within the harness tolerances."""
import numpy as np
import pytest
import torch

import synth
from harness import FULL, RING, ROLL, SLIDING, assert_bits_equal, assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu
D = synth.HEAD_DIM


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _ctx(hd, types, Hq, Hkv, B, max_context, kv="bf16", layout=0):
    return hd.hybrid_decode_init(hd.Config(layer_types=types, num_q_heads=Hq, num_kv_heads=Hkv, max_batch=B,
                                           max_context=max_context, cache_layout=layout,
                                           kv_dtype=hd.HD_KV_FP8_E4M3 if kv == "fp8" else hd.HD_KV_BF16))


class TokenLayer:
    """Seeded inputs of one layer of a T-token step."""

    def __init__(self, rng, t, B, T, Hq, Hkv, cap, context, kv, sink, with_gate):
        written = np.minimum(context, cap)
        self.t, self.kv = t, kv
        self.q = synth.normal_bf16(rng, (B, T, Hq, D))
        self.k = synth.normal_bf16(rng, (B, T, Hkv, D))
        self.v = synth.normal_bf16(rng, (B, T, Hkv, D))
        self.k_scale = self.v_scale = None
        if kv == "fp8":
            self.k_scale, self.v_scale = synth.kv_scales(rng, Hkv), synth.kv_scales(rng, Hkv)
            self.kc = synth.cache_with_history_fp8(rng, B, Hkv, cap, written, self.k_scale)
            self.vc = synth.cache_with_history_fp8(rng, B, Hkv, cap, written, self.v_scale)
        else:
            self.kc = synth.cache_with_history(rng, B, Hkv, cap, written)
            self.vc = synth.cache_with_history(rng, B, Hkv, cap, written)
        self.sink = sink
        self.gate = torch.from_numpy(rng.standard_normal((B, T, Hq)).astype(np.float32) * 2) if with_gate else None

    def oracle(self, orc, context, layout):
        rot, theta = synth.ROPE[self.t]
        kc, vc = synth.bits(self.kc), synth.bits(self.vc)
        r = orc.decode_tokens(layer_type=self.t, layout=layout if self.t == SLIDING else 0, window=synth.WINDOW,
                              rotary_dim=rot, rope_theta=theta, context=context, q=synth.bits(self.q),
                              k=synth.bits(self.k), v=synth.bits(self.v), kcache=kc, vcache=vc,
                              sink=None if self.sink is None else self.sink.numpy(),
                              gate=None if self.gate is None else self.gate.numpy(),
                              k_scale=None if self.k_scale is None else self.k_scale.numpy(),
                              v_scale=None if self.v_scale is None else self.v_scale.numpy())
        r["kcache"], r["vcache"] = kc, vc
        return r

    def device(self, hd):
        dev = torch.device("cuda")
        self.kd, self.vd = self.kc.to(dev), self.vc.to(dev)
        if self.kv == "fp8":   # the descriptor holds raw pointers: keep the device scales
            self.scales_dev = (self.k_scale.to(dev), self.v_scale.to(dev))
            self.cache = hd.kv_cache(self.kd, self.vd, *self.scales_dev)
        else:
            self.cache = hd.kv_cache(self.kd, self.vd)
        B, T, Hq, _ = self.q.shape
        self.out = torch.empty(B, T, Hq, D, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(B, T, Hq, dtype=torch.float32, device=dev)
        self.keep = [x.to(dev) if x is not None else None for x in (self.q, self.k, self.v, self.sink, self.gate)]
        q, k, v, sink, gate = self.keep
        return hd.layer_io(q, k, v, self.cache, sink, self.out, self.lse, gate=gate)


def run_case(hd, orc, types, T, Hq, Hkv, context, kv="bf16", seed=0, with_gate=True, max_context=None,
             fuse=True, layout=RING, consumer=None):
    rng = synth.generator(seed)
    B = len(context)
    context = np.asarray(context, np.int32)
    max_context = max_context or int(context.max()) + T
    ctx = _ctx(hd, types, Hq, Hkv, B, max_context, kv, layout=layout)
    hd.hybrid_decode_set_step_fusion(ctx, fuse)
    if consumer is not None:
        hd.hybrid_decode_set_consumer(ctx, consumer)
    sink = synth.sink_vector(rng, ("normal", 1.0, 0.0), Hq)
    window = synth.WINDOW - 1 if layout == RING else synth.WINDOW
    layers = [TokenLayer(rng, t, B, T, Hq, Hkv, window if t == SLIDING else max_context + 1, context, kv, sink,
                         with_gate) for t in types]
    refs = [L.oracle(orc, context, layout) for L in layers]
    ios = [L.device(hd) for L in layers]
    hd.decode_step_tokens(ctx, torch.from_numpy(context).cuda(), ios, B, T)
    torch.cuda.synchronize()
    assert hd.hybrid_decode_device_errors(ctx) == 0
    for i, (L, ref) in enumerate(zip(layers, refs)):
        assert_out_close(L.out, ref["out"], f"layer {i} out")
        assert_lse_close(L.lse, ref["lse"], f"layer {i} lse")
        assert_bits_equal(L.kd, ref["kcache"], f"layer {i} K cache")
        assert_bits_equal(L.vd, ref["vcache"], f"layer {i} V cache")
    ctx.close()


RING_FULL_CONTEXTS = [0, 1, 300, 505, 509, 510, 511, 512, 700, 1021, 1500, 3000]


@pytest.mark.parametrize("T", [2, 3, 4, 8])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_tokens_ring_and_full(hd, orc, T, g):
    """A [sliding ring, full] pair with T tokens across the ring's wrap points."""
    Hkv = 2
    run_case(hd, orc, [SLIDING, FULL], T, g * Hkv, Hkv, RING_FULL_CONTEXTS, seed=700 + 10 * T + g)


ROLL_CONTEXTS = [0, 1, 300, 505, 508, 509, 510, 511, 512, 513, 700, 1500]


@pytest.mark.parametrize("fuse", [True, False])
@pytest.mark.parametrize("T", [2, 3, 4, 8])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_tokens_roll_and_full(hd, orc, T, g, fuse):
    """A [sliding roll, full] pair with T tokens while the rolled window fills up
    and once it is full: each token sees its own window (the window is read once,
    before it shifts by the entries that leave it), and the window ends as after
    T single-token steps.  Step fusion on (one grid) and off (one kernel per layer)."""
    Hkv = 2
    run_case(hd, orc, [SLIDING, FULL], T, g * Hkv, Hkv, ROLL_CONTEXTS, seed=1300 + 10 * T + g, fuse=fuse,
             layout=ROLL)


@pytest.mark.parametrize("T", [2, 5])
def test_tokens_roll_fp8(hd, orc, T):
    run_case(hd, orc, [SLIDING, FULL], T, 8, 2, ROLL_CONTEXTS, kv="fp8", seed=1400 + T, layout=ROLL)


def test_tokens_roll_28_layer_step(hd, orc):
    run_case(hd, orc, synth.SPARK_LAYER_TYPES, 4, 8, 2, [510, 1500, 3], seed=1410, layout=ROLL)


@pytest.mark.parametrize("T", [2, 4, 5])
@pytest.mark.parametrize("g", [2, 4, 8])
def test_tokens_fp8(hd, orc, T, g):
    Hkv = 2
    run_case(hd, orc, [SLIDING, FULL], T, g * Hkv, Hkv, RING_FULL_CONTEXTS, kv="fp8", seed=800 + 10 * T + g)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("T", [3, 4])
def test_tokens_kernel_per_layer(hd, orc, kv, T):
    """Step fusion off: each layer's passes run as their own kernels."""
    run_case(hd, orc, [SLIDING, FULL], T, 8, 2, RING_FULL_CONTEXTS, kv=kv, seed=950 + T, fuse=False)


def test_tokens_one_equals_decode_step(hd, orc):
    """T = 1 is the single-token step (same kernel path, same results)."""
    run_case(hd, orc, [SLIDING, FULL, SLIDING], 1, 8, 2, [5, 600, 2000], seed=901)


def test_tokens_long_context_many_chunks(hd, orc):
    run_case(hd, orc, [FULL], 4, 8, 2, [40000, 39000 - 7], seed=902, with_gate=False)


def test_tokens_28_layer_step(hd, orc):
    run_case(hd, orc, synth.SPARK_LAYER_TYPES, 4, 8, 2, [700, 1500, 3], seed=903)


# The tensor-memory consumer runs passes of 16 or 32 rows (g x tokens per pass) on
# tcgen05 with 64-key stages; other passes of the same call run mma.sync.
@pytest.mark.parametrize("fuse", [True, False])
@pytest.mark.parametrize("T,g", [(4, 4), (2, 8), (8, 2), (8, 4), (4, 8), (8, 8), (3, 8)])
def test_tokens_tensor_memory_consumer(hd, orc, T, g, fuse):
    Hkv = 2
    run_case(hd, orc, [SLIDING, FULL], T, g * Hkv, Hkv, RING_FULL_CONTEXTS, seed=1500 + 10 * T + g, fuse=fuse,
             consumer=hd.HD_CONSUMER_TENSOR_MEMORY)


@pytest.mark.parametrize("T,g", [(4, 4), (8, 4), (4, 8)])
def test_tokens_tensor_memory_roll(hd, orc, T, g):
    run_case(hd, orc, [SLIDING, FULL], T, 2 * g, 2, ROLL_CONTEXTS, seed=1600 + 10 * T + g, layout=ROLL,
             consumer=hd.HD_CONSUMER_TENSOR_MEMORY)


def test_tokens_tensor_memory_long_context_and_28_layers(hd, orc):
    run_case(hd, orc, [FULL], 4, 8, 2, [40000, 39000 - 7], seed=1610, with_gate=False,
             consumer=hd.HD_CONSUMER_TENSOR_MEMORY)
    run_case(hd, orc, [FULL], 4, 16, 2, [40000, 39000 - 7], seed=1612, with_gate=False,
             consumer=hd.HD_CONSUMER_TENSOR_MEMORY)
    run_case(hd, orc, synth.SPARK_LAYER_TYPES, 4, 8, 2, [700, 1500, 3], seed=1611,
             consumer=hd.HD_CONSUMER_TENSOR_MEMORY)


def test_tokens_tensor_memory_fp8_falls_back(hd, orc):
    """E4M3 caches have no tensor-memory pass: the same call runs mma.sync."""
    run_case(hd, orc, [SLIDING, FULL], 4, 8, 2, RING_FULL_CONTEXTS, kv="fp8", seed=1620,
             consumer=hd.HD_CONSUMER_TENSOR_MEMORY)


def test_tokens_match_sequential_gpu_steps(hd):
    """A 4-token step and four single-token steps on the GPU write the same cache
    bits and give outputs equal to rounding."""
    rng = synth.generator(904)
    B, T, Hq, Hkv = 3, 4, 8, 2
    context = np.array([509, 1200, 40], np.int32)
    types = [SLIDING, FULL]
    sink = synth.sink_vector(rng, ("normal", 1.0, 0.0), Hq)
    layers = [TokenLayer(rng, t, B, T, Hq, Hkv, 511 if t == SLIDING else 1300, context, "bf16", sink, False)
              for t in types]
    ctx = _ctx(hd, types, Hq, Hkv, B, 1299)
    ios = [L.device(hd) for L in layers]
    kc0 = [(L.kd.clone(), L.vd.clone()) for L in layers]
    hd.decode_step_tokens(ctx, torch.from_numpy(context).cuda(), ios, B, T)
    seq_out = []
    for i, L in enumerate(layers):  # restore the caches, then one token at a time
        L.seq_k, L.seq_v = kc0[i][0].clone(), kc0[i][1].clone()
    for t in range(T):
        step_ios, outs = [], []
        for L in layers:
            q, k, v, s, _ = L.keep
            out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
            lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
            qt, kt, vt = q[:, t].contiguous(), k[:, t].contiguous(), v[:, t].contiguous()   # kept alive below
            step_ios.append(hd.layer_io(qt, kt, vt, hd.kv_cache(L.seq_k, L.seq_v), s, out, lse))
            outs.append((out, lse, step_ios[-1], qt, kt, vt))
        hd.decode_step(ctx, torch.from_numpy(context + t).cuda(), step_ios, B)
        torch.cuda.synchronize()
        seq_out.append(outs)
    assert hd.hybrid_decode_device_errors(ctx) == 0
    for i, L in enumerate(layers):
        assert_bits_equal(L.kd, synth.bits(L.seq_k), f"layer {i} K cache")   # bits: unwritten slots are NaN
        assert_bits_equal(L.vd, synth.bits(L.seq_v), f"layer {i} V cache")
        for t in range(T):
            a, b = L.out[:, t].float(), seq_out[t][i][0].float()
            assert torch.all((a - b).abs() <= 1e-2 + 1e-2 * b.abs()), f"layer {i} token {t}"
            assert torch.all((L.lse[:, t] - seq_out[t][i][1]).abs() <= 1e-4)
    ctx.close()


def test_tokens_unsupported_paths(hd):
    """Several tokens need the tensor-core consumer."""
    rng = synth.generator(905)
    B, T, Hq, Hkv = 1, 2, 8, 2
    ctx = _ctx(hd, [FULL], Hq, Hkv, B, 100)
    hd.hybrid_decode_set_consumer(ctx, hd.HD_CONSUMER_CUDA_CORE)
    L = TokenLayer(rng, FULL, B, T, Hq, Hkv, 101, np.array([10], np.int32), "bf16", None, False)
    with pytest.raises(hd.HDError) as e:
        hd.decode_step_tokens(ctx, torch.tensor([10], dtype=torch.int32, device="cuda"), [L.device(hd)], B, T)
    assert e.value.status == 2
    ctx.close()
