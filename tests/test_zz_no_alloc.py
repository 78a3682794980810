"""The allocation-free full-layer entry point, checked against the fp64 oracle
and against the regular entry point.

decode_attn_full_static_scratch serves callers that cannot allocate device
memory while running (a plugin inside a runtime that owns every allocation,
a serving loop where cudaMalloc/cudaFree could synchronise the device): it
needs no context and keeps its split-K scratch in a fixed array inside the
library.  Its inputs here come straight from the oracle (the rotated q and
the caches after the new entry was appended), so no other GPU call feeds it.
Called twice in a row through the C ABI, it must match the oracle and
decode_attn_full within the parity tolerances; a call whose scratch would
not fit the array is refused before anything is launched.  This file is
collected last on purpose."""
import numpy as np
import pytest
import torch

import synth
from harness import FULL, LSE_ATOL, OUT_ATOL, OUT_RTOL, LayerCase, assert_lse_close, assert_out_close, oracle_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16)


CASES = {
    # one CTA per SM or fewer: the deep-ring plan, group 4, a quarter of the sinks -inf
    "b6_g4": dict(seed=77, B=6, Hq=8, Hkv=2, contexts=[0, 1, 777, 4095, 8191, 9000], sink=("normal", 2.0 ** 0.5, 0.25)),
    # more CTAs than SMs (three-stage plan, several chunks per sequence), group 8, -inf sinks
    "b64_g8": dict(seed=78, B=64, Hq=16, Hkv=2, contexts=None, sink=("normal", 2.0 ** 0.5, 0.25)),
    # groups 1 and 2, no sink
    "b3_g1": dict(seed=79, B=3, Hq=2, Hkv=2, contexts=[5, 2047, 2048], sink=None),
    "b5_g2": dict(seed=80, B=5, Hq=4, Hkv=2, contexts=[0, 64, 511, 3000, 6000], sink=("normal", 1.0, 0.0)),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_static_scratch_matches_oracle_and_decode_attn_full_twice(hd, orc, name):
    spec = CASES[name]
    rng = synth.generator(spec["seed"])
    B, Hq, Hkv, D = spec["B"], spec["Hq"], spec["Hkv"], synth.HEAD_DIM
    contexts = (np.asarray(spec["contexts"], np.int32) if spec["contexts"] is not None
                else np.concatenate([rng.integers(1, 513, 8), rng.integers(2000, 4097, B - 8)]).astype(np.int32))
    max_ctx = int(contexts.max())
    sink = None if spec["sink"] is None else synth.sink_vector(rng, spec["sink"], Hq)
    case = LayerCase(rng, B, Hq, Hkv, max_ctx + 1, contexts, sink=sink)
    ref = oracle_layer(orc, case, FULL, 0)

    # The oracle's rotated q and its caches after the step (the new entry at index c).
    dev = torch.device("cuda")
    context = torch.from_numpy(contexts).to(dev)
    q_rot = torch.from_numpy(ref["qrot"].astype(np.float32)).to(dev)
    kc, vc = _bf16(ref["kcache"]).to(dev), _bf16(ref["vcache"]).to(dev)
    cache = hd.kv_cache(kc, vc)
    sink_d = None if sink is None else sink.to(dev)

    runs = []
    for call in range(2):
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev)
        hd.decode_attn_full_static_scratch(Hkv, context, max_ctx, q_rot, cache, sink_d, out, lse)
        torch.cuda.synchronize()
        assert_out_close(out, ref["out"], f"call {call}: out")
        assert_lse_close(lse, ref["lse"], f"call {call}: lse")
        runs.append((out, lse))

    # The regular entry point on the same inputs (its own context and workspace).
    ctx = hd.hybrid_decode_init(hd.Config(layer_types=[FULL], num_q_heads=Hq, num_kv_heads=Hkv,
                                          max_batch=B, max_context=max_ctx))
    ref_out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    ref_lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    hd.decode_attn_full(ctx, 0, context, q_rot, cache, sink_d, ref_out, ref_lse)
    torch.cuda.synchronize()
    assert hd.hybrid_decode_device_errors(ctx) == 0
    ctx.close()
    r = ref_out.float()
    for call, (out, lse) in enumerate(runs):
        g = out.float()
        assert torch.all((g - r).abs() <= OUT_ATOL + OUT_RTOL * r.abs()), f"call {call}: out differs from decode_attn_full"
        assert torch.all((lse - ref_lse).abs() <= LSE_ATOL), f"call {call}: lse differs from decode_attn_full"
    # the caches are inputs only
    assert np.array_equal(synth.bits(kc), ref["kcache"]) and np.array_equal(synth.bits(vc), ref["vcache"])


def test_static_scratch_refuses_sizes_beyond_its_array(hd):
    """A call whose split-K scratch exceeds the array is refused before any launch.
    The cache buffer really holds every row the descriptor claims (K and V share
    it), so nothing here could read past an allocation."""
    dev = torch.device("cuda")
    B, Hq, Hkv, D, max_ctx = 16, 64, 8, 256, 131071
    nbytes, _, _, st = hd.decode_attn_full_static_scratch_plan(B, Hq, Hkv, max_ctx,
                                                               torch.cuda.get_device_properties(dev).multi_processor_count)
    assert st == 3 and nbytes > hd.HD_STATIC_SCRATCH_BYTES
    kv = torch.empty(B, Hkv, max_ctx + 1, D, dtype=torch.bfloat16, device=dev)   # 8.6 GB, honest extent
    context = torch.zeros(B, dtype=torch.int32, device=dev)
    q_rot = torch.zeros(B, Hq, D, dtype=torch.float32, device=dev)
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    cache = hd.kv_cache(kv, kv)
    with pytest.raises(hd.HDError) as e:
        hd.decode_attn_full_static_scratch(Hkv, context, max_ctx, q_rot, cache, None, out, lse)
    assert e.value.status == 3
    del kv
    torch.cuda.empty_cache()
