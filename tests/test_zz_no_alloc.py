"""The allocation-free full-layer entry point against the regular one.

decode_attn_full_static_scratch serves callers that cannot allocate device
memory while running (a plugin inside a runtime that owns every allocation,
a serving loop where cudaMalloc/cudaFree could synchronise the device): it
needs no context and keeps its split-K scratch in a fixed array inside the
library.  Called twice in a row through the C ABI, it must match
decode_attn_full within the parity tolerances; sizes beyond its scratch are
refused before any launch.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import synth
from harness import FULL, LSE_ATOL, OUT_ATOL, OUT_RTOL, LayerCase

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def test_static_scratch_matches_decode_attn_full_twice(hd):
    rng = synth.generator(77)
    B, Hq, Hkv, D, max_ctx = 6, 8, 2, 256, 9000
    contexts = np.array([0, 1, 777, 4095, 8191, 9000], np.int32)
    ctx = hd.hybrid_decode_init(hd.Config(layer_types=[FULL], num_q_heads=Hq, num_kv_heads=Hkv,
                                          max_batch=B, max_context=max_ctx))
    case = LayerCase(rng, B, Hq, Hkv, max_ctx + 1, contexts,
                     sink=synth.sink_vector(rng, ("normal", 2.0 ** 0.5, 0.25), Hq))
    dev = torch.device("cuda")
    context = torch.from_numpy(contexts).to(dev)
    kc, vc = case.kc.to(dev), case.vc.to(dev)
    cache = hd.kv_cache(kc, vc)
    sink = case.sink.to(dev)
    q_rot = torch.empty(B, Hq, D, dtype=torch.float32, device=dev)
    hd.rope_append_kv(ctx, 0, context, case.q.to(dev), case.k.to(dev), case.v.to(dev), q_rot, cache)
    ref_out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    ref_lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    hd.decode_attn_full(ctx, 0, context, q_rot, cache, sink, ref_out, ref_lse)
    torch.cuda.synchronize()
    assert hd.hybrid_decode_device_errors(ctx) == 0
    for call in range(2):
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev)
        hd.decode_attn_full_static_scratch(Hkv, context, max_ctx, q_rot, cache, sink, out, lse)
        torch.cuda.synchronize()
        r, g = ref_out.float(), out.float()
        assert torch.isfinite(g).all(), f"call {call}: non-finite output"
        assert torch.all((g - r).abs() <= OUT_ATOL + OUT_RTOL * r.abs()), f"call {call}: out differs"
        assert torch.all((lse - ref_lse).abs() <= LSE_ATOL), f"call {call}: lse differs"
    ctx.close()


def test_static_scratch_refuses_sizes_beyond_its_array(hd):
    dev = torch.device("cuda")
    B, Hq, Hkv, D, max_ctx = 256, 16, 2, 256, 131072   # needs far more than the 64 MiB array
    context = torch.zeros(B, dtype=torch.int32, device=dev)
    q_rot = torch.zeros(B, Hq, D, dtype=torch.float32, device=dev)
    k = torch.zeros(B, Hkv, 16, D, dtype=torch.bfloat16, device=dev)
    cache = hd.hd_kv_cache(k.data_ptr(), k.data_ptr(), Hkv * (max_ctx + 1) * D, max_ctx + 1)
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    with pytest.raises(hd.HDError) as e:
        hd.decode_attn_full_static_scratch(Hkv, context, max_ctx, q_rot, cache, None, out, lse)
    assert e.value.status == 3
