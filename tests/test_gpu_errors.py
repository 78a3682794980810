"""Error paths that reach the GPU: rejected on the host before any launch, or
detected by the kernels, which skip the offending sequence (no out-of-bounds
access) and record a bit in the context's device error word.  Nothing here
faults or hangs a GPU."""
import numpy as np
import pytest
import torch

import synth
from harness import FULL, RING, SLIDING, LayerCase, assert_lse_close, assert_out_close, oracle_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _ctx(hd, types, **kw):
    base = dict(layer_types=types, max_batch=4, max_context=1024)
    base.update(kw)
    return hd.hybrid_decode_init(hd.Config(**base))


def _bufs(B, Hq=8, D=256):
    dev = "cuda"
    return (torch.empty(B, Hq, D, dtype=torch.float32, device=dev),
            torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev),
            torch.empty(B, Hq, dtype=torch.float32, device=dev))


def test_device_detects_bad_contexts_and_serves_the_rest(hd, orc):
    rng = synth.generator(5)
    ctx = _ctx(hd, [FULL])
    context = np.array([10, 150, -3, 60], np.int32)   # 150 >= capacity 101; -3 negative
    case = LayerCase(rng, 4, 8, 2, 101, np.clip(context, 0, 100),
                     sink=synth.sink_vector(rng, ("normal", 1.0, 0.0), 8))
    case.context = context
    qrot, out, lse = _bufs(4)
    kd, vd = case.kc.cuda(), case.vc.cuda()
    cache = hd.kv_cache(kd, vd)
    ctx_d = torch.from_numpy(context).cuda()
    hd.rope_append_kv(ctx, 0, ctx_d, case.q.cuda(), case.k.cuda(), case.v.cuda(), qrot, cache)
    hd.decode_attn_full(ctx, 0, ctx_d, qrot, cache, case.sink.cuda(), out, lse, max_context_hint=100)
    flags = hd.hybrid_decode_device_errors(ctx)
    assert flags & 2 and flags & 1, f"flags {flags:#x}"
    assert hd.hybrid_decode_device_errors(ctx) == 0  # cleared by the read
    assert torch.isnan(out[1].float()).all() and torch.isnan(out[2].float()).all()
    good = [0, 3]
    sub = LayerCase(rng, 2, 8, 2, 101, context[good], sink=case.sink)
    sub.q, sub.k, sub.v = case.q[good], case.k[good], case.v[good]
    sub.kc, sub.vc = case.kc[good].contiguous(), case.vc[good].contiguous()
    ref = oracle_layer(orc, sub, FULL, 0)
    assert_out_close(out[good], ref["out"])
    assert_lse_close(lse[good], ref["lse"])


def test_context_beyond_max_context_is_flagged(hd):
    rng = synth.generator(6)
    ctx = _ctx(hd, [SLIDING])
    case = LayerCase(rng, 1, 8, 2, 511, [2000], written=[511])
    qrot, out, lse = _bufs(1)
    cache = hd.kv_cache(case.kc.cuda(), case.vc.cuda())
    ctx_d = torch.tensor([2000], dtype=torch.int32, device="cuda")
    hd.rope_append_kv(ctx, 0, ctx_d, case.q.cuda(), case.k.cuda(), case.v.cuda(), qrot, cache)
    hd.decode_attn_sliding(ctx, 0, ctx_d, qrot, cache, None, out, lse)
    assert hd.hybrid_decode_device_errors(ctx) & 4
    assert torch.isnan(lse).all()


def test_host_rejections(hd):
    rng = synth.generator(7)
    ctx = _ctx(hd, [SLIDING, FULL], max_batch=2)
    case = LayerCase(rng, 3, 8, 2, 511, [5, 5, 5])
    qrot, out, lse = _bufs(3)
    ring = hd.kv_cache(case.kc.cuda(), case.vc.cuda())
    ctx3 = torch.full((3,), 5, dtype=torch.int32, device="cuda")
    with pytest.raises(hd.HDError) as e:   # batch 3 > max_batch 2
        hd.decode_attn_sliding(ctx, 0, ctx3, qrot, ring, None, out, lse)
    assert e.value.status == 3
    ctx2, q2 = ctx3[:2], qrot[:2]
    with pytest.raises(hd.HDError) as e:   # full-layer call on a sliding layer
        hd.decode_attn_full(ctx, 0, ctx2, q2, ring, None, out[:2], lse[:2])
    assert e.value.status == 5
    full_small = hd.kv_cache(case.kc[:2].cuda(), case.vc[:2].cuda())   # capacity 511 < 1025
    with pytest.raises(hd.HDError) as e:
        hd.decode_attn_full(ctx, 1, ctx2, q2, full_small, None, out[:2], lse[:2])
    assert e.value.status == 3
    wrong = LayerCase(rng, 2, 8, 2, 512, [5, 5])   # a ring must hold window-1 = 511 entries
    with pytest.raises(hd.HDError) as e:
        hd.decode_attn_sliding(ctx, 0, ctx2, q2, hd.kv_cache(wrong.kc.cuda(), wrong.vc.cuda()),
                               None, out[:2], lse[:2])
    assert e.value.status == 3
    misaligned = qrot.view(-1)[1:1 + 2 * 8 * 256].view(2, 8, 256)
    with pytest.raises(hd.HDError) as e:
        hd.decode_attn_sliding(ctx, 0, ctx2, misaligned, ring, None, out[:2], lse[:2])
    assert e.value.status == 1
    with pytest.raises(hd.HDError) as e:   # hint beyond max_context
        hd.decode_attn_full(ctx, 1, ctx2, q2, ring, None, out[:2], lse[:2], max_context_hint=5000)
    assert e.value.status == 3


def test_sink_checks_mirror_the_page(hd):
    ctx = _ctx(hd, [SLIDING])
    rng = synth.generator(8)
    case = LayerCase(rng, 1, 8, 2, 511, [5])
    qrot, out, lse = _bufs(1)
    cache = hd.kv_cache(case.kc.cuda(), case.vc.cuda())
    ctx_d = torch.tensor([5], dtype=torch.int32, device="cuda")
    for bad in (torch.zeros(8, dtype=torch.float16, device="cuda"),   # not fp32
                torch.zeros(7, device="cuda"),                         # wrong head count
                torch.zeros(8)):                                       # other device
        with pytest.raises(ValueError):
            hd.decode_attn_sliding(ctx, 0, ctx_d, qrot, cache, bad, out, lse)


def test_lost_copy_times_out_and_the_context_recovers(hd, orc):
    """A copy that never arrives: the bounded waits run out (about one second),
    the kernel reports HD_DEVERR_WAIT_TIMEOUT and returns; the same context then
    gives correct results again."""
    import time
    rng = synth.generator(9)
    ctx = _ctx(hd, [FULL], max_batch=2, max_context=1024)
    case = LayerCase(rng, 2, 8, 2, 1025, [300, 900], sink=synth.sink_vector(rng, ("normal", 1.0, 0.0), 8))
    dev = torch.device("cuda")
    context = torch.from_numpy(case.context).to(dev)
    kc, vc = case.kc.to(dev), case.vc.to(dev)
    cache = hd.kv_cache(kc, vc)
    qrot, out, lse = _bufs(2)
    hd.rope_append_kv(ctx, 0, context, case.q.to(dev), case.k.to(dev), case.v.to(dev), qrot, cache)
    hd.hybrid_decode_inject_lost_copy(ctx, 1)
    t0 = time.time()
    hd.decode_attn_full(ctx, 0, context, qrot, cache, case.sink.to(dev), out, lse)
    flags = hd.hybrid_decode_device_errors(ctx)
    elapsed = time.time() - t0
    assert flags & 8, f"expected a wait timeout, flags {flags:#x}"
    assert 0.5 < elapsed < 30.0, elapsed
    hd.hybrid_decode_inject_lost_copy(ctx, -1)
    hd.decode_attn_full(ctx, 0, context, qrot, cache, case.sink.to(dev), out, lse)
    assert hd.hybrid_decode_device_errors(ctx) == 0
    ref = oracle_layer(orc, case, FULL, 0)
    assert_out_close(out, ref["out"])
    assert_lse_close(lse, ref["lse"])
