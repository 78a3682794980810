"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (bench.Workload + decode_step): the whole step runs on the GPU, and the
oracle recomputes every layer for a few sampled sequences (shortest, median,
longest).  Inputs are copied to the host before the step, so the oracle sees
exactly the GPU's inputs; after the step each sampled sequence's caches must
equal the oracle's caches bit for bit (the written entry and everything else).
"""
import numpy as np
import pytest
import torch

import bench
import synth
from harness import assert_bits_equal, assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _samples(context, k=3):
    order = np.argsort(context, kind="stable")
    picks = [order[0], order[len(order) // 2], order[-1]][:k]
    return sorted(set(int(b) for b in picks))


def _snapshot(wl, samples):
    """Host copies of every layer's inputs for the sampled sequences."""
    snap = []
    for L in wl.layers:
        snap.append({b: dict(q=synth.bits(L["q"][b:b + 1]), k=synth.bits(L["k"][b:b + 1]),
                             v=synth.bits(L["v"][b:b + 1]), kc=synth.bits(L["kc"][b:b + 1]),
                             vc=synth.bits(L["vc"][b:b + 1])) for b in samples})
    return snap


def _check_against_oracle(hd, orc, wl, snap, samples, layers=None):
    sink = None if wl.sink is None else wl.sink.cpu().numpy()
    layout = synth.LAYOUT_ROLL if wl.layout == synth.LAYOUT_ROLL else synth.LAYOUT_RING
    for i, t in enumerate(wl.types):
        if layers is not None and i not in layers:
            continue
        rot, theta = synth.ROPE[t]
        L = wl.layers[i]
        for b in samples:
            s = snap[i][b]
            scales = {}
            if wl.kv == "fp8":
                scales = dict(k_scale=L["k_scale"].cpu().numpy(), v_scale=L["v_scale"].cpu().numpy())
            ref = orc.decode_layer(layer_type=t, layout=layout if t == synth.SLIDING else 0,
                                   window=synth.WINDOW, rotary_dim=rot, rope_theta=theta,
                                   context=wl.context[b:b + 1], q=s["q"], k=s["k"], v=s["v"],
                                   kcache=s["kc"], vcache=s["vc"], sink=sink, **scales)
            assert_out_close(L["out"][b:b + 1], ref["out"], f"layer {i} seq {b} out")
            assert_lse_close(L["lse"][b:b + 1], ref["lse"], f"layer {i} seq {b} lse")
            assert_bits_equal(L["kc"][b:b + 1], s["kc"], f"layer {i} seq {b} K cache")
            assert_bits_equal(L["vc"][b:b + 1], s["vc"], f"layer {i} seq {b} V cache")


def _run(hd, wl):
    wl.step()
    torch.cuda.synchronize()
    assert hd.hybrid_decode_device_errors(wl.ctx) == 0


def test_step28_batch64_contexts_512_to_32768(hd, orc):
    """The benchmark's own workload: 28 layers, batch 64, c ~ U[512, 32768], sink."""
    wl = bench.Workload("step28_b64_c512_32768", torch.device("cuda"), seed=0)
    samples = _samples(wl.context)
    snap = _snapshot(wl, samples)
    _run(hd, wl)
    _check_against_oracle(hd, orc, wl, snap, samples)
    wl.ctx.close()


def test_step28_batch64_e4m3_caches(hd, orc):
    """The same workload with E4M3 caches (per-kv-head scales), as bench.py --kv fp8 runs it."""
    wl = bench.Workload("step28_b64_c512_32768", torch.device("cuda"), seed=0, kv="fp8")
    samples = _samples(wl.context)
    snap = _snapshot(wl, samples)
    _run(hd, wl)
    _check_against_oracle(hd, orc, wl, snap, samples)
    wl.ctx.close()


def test_step28_batch64_roll_layout(hd, orc):
    """The same workload with rolled sliding windows, shifted inside the step grid."""
    wl = bench.Workload("step28_b64_c512_32768", torch.device("cuda"), seed=0, layout=synth.LAYOUT_ROLL)
    samples = _samples(wl.context)
    snap = _snapshot(wl, samples)
    _run(hd, wl)
    _check_against_oracle(hd, orc, wl, snap, samples)
    wl.ctx.close()


def test_step28_batch1_context_4096(hd, orc):
    wl = bench.Workload("step28_b1_c4096", torch.device("cuda"), seed=0)
    snap = _snapshot(wl, [0])
    _run(hd, wl)
    _check_against_oracle(hd, orc, wl, snap, [0])
    wl.ctx.close()


def test_long_context_131072_full_layers(hd, orc):
    """7 full layers, batch 4 at context 131072 (split into >= 64 chunks)."""
    wl = bench.Workload("full7_b4_c131072", torch.device("cuda"), seed=0)
    ck, nc = hd.hd_plan_split(4, 2, 131072, torch.cuda.get_device_properties(0).multi_processor_count)
    assert nc >= 64
    snap = _snapshot(wl, [0, 3])
    _run(hd, wl)
    _check_against_oracle(hd, orc, wl, snap, [0], layers=range(7))
    _check_against_oracle(hd, orc, wl, snap, [3], layers=[0, 6])
    wl.ctx.close()


def test_group8_batch256_ring_and_roll(hd, orc):
    """16 q / 2 kv heads, 230 sequences at 8192 and 26 short ones, sink N(0, variance 2)
    with a quarter of the heads at -inf; the ring and the roll layouts run on the same
    window contents and must agree with each other and with the oracle."""
    dev = torch.device("cuda")
    ring = bench.Workload("step28_b256_g8_mixed", dev, seed=0, layout=synth.LAYOUT_RING)
    roll = bench.Workload("step28_b256_g8_mixed", dev, seed=0, layout=synth.LAYOUT_ROLL)
    ctx_d = ring.context_d.long()
    for Lr, Ll, t in zip(ring.layers, roll.layers, ring.types):
        for key in ("q", "k", "v"):
            Ll[key].copy_(Lr[key])
        if t == synth.FULL:
            Ll["kc"].copy_(Lr["kc"])
            Ll["vc"].copy_(Lr["vc"])
            continue
        # Roll index i holds position c-512+i; the ring holds position p at slot p mod 511.
        # (Index 0 holds position c-512, which the ring has evicted; the roll step drops
        # it once the window is full, so any value serves there.)
        i = torch.arange(512, device=dev)
        pos = ctx_d[:, None] - 512 + i[None, :]
        slot = torch.where(ctx_d[:, None] >= 512, torch.remainder(pos, 511), i[None, :].clamp(max=510))
        idx = slot[:, None, :, None].expand(-1, ring.Hkv, -1, synth.HEAD_DIM)
        Ll["kc"].copy_(torch.gather(Lr["kc"], 2, idx))
        Ll["vc"].copy_(torch.gather(Lr["vc"], 2, idx))
    samples = _samples(ring.context)
    snap_ring = _snapshot(ring, samples)
    snap_roll = _snapshot(roll, samples)
    _run(hd, ring)
    _run(hd, roll)
    for i, (Lr, Ll) in enumerate(zip(ring.layers, roll.layers)):
        a, b = Lr["out"].float(), Ll["out"].float()
        assert torch.all((a - b).abs() <= 2e-2 + 2e-2 * a.abs()), f"layer {i}: ring and roll differ"
        assert torch.all((Lr["lse"] - Ll["lse"]).abs() <= 1e-3), f"layer {i}: ring and roll lse differ"
    _check_against_oracle(hd, orc, ring, snap_ring, samples)
    _check_against_oracle(hd, orc, roll, snap_roll, samples, layers=[0, 1, 3])
    ring.ctx.close()
    roll.ctx.close()


def _check_tokens_against_oracle(orc, wl, snap, samples):
    """Every layer of a multi-token step for the sampled sequences: the oracle's
    T single-token steps in order (its caches updated in place)."""
    sink = None if wl.sink is None else wl.sink.cpu().numpy()
    layout = synth.LAYOUT_ROLL if wl.layout == synth.LAYOUT_ROLL else synth.LAYOUT_RING
    for i, t in enumerate(wl.types):
        rot, theta = synth.ROPE[t]
        L = wl.layers[i]
        for b in samples:
            s = snap[i][b]
            kc, vc = s["kc"].copy(), s["vc"].copy()
            ref = orc.decode_tokens(layer_type=t, layout=layout if t == synth.SLIDING else 0, window=synth.WINDOW,
                                    rotary_dim=rot, rope_theta=theta, context=wl.context[b:b + 1], q=s["q"],
                                    k=s["k"], v=s["v"], kcache=kc, vcache=vc, sink=sink, gate=None,
                                    k_scale=None, v_scale=None)
            assert_out_close(L["out"][b:b + 1], ref["out"], f"layer {i} seq {b} out")
            assert_lse_close(L["lse"][b:b + 1], ref["lse"], f"layer {i} seq {b} lse")
            assert_bits_equal(L["kc"][b:b + 1], kc, f"layer {i} seq {b} K cache")
            assert_bits_equal(L["vc"][b:b + 1], vc, f"layer {i} seq {b} V cache")


def test_step28_batch64_eight_tokens(hd, orc):
    """The benchmark workload decoding 8 tokens per sequence, as bench.py's
    multi_token T = 8 runs it: 32 query rows per kv head, one tcgen05 pass per
    layer over the whole cache."""
    wl = bench.Workload("step28_b64_c512_32768", torch.device("cuda"), seed=0, tokens=8)
    samples = _samples(wl.context)
    snap = _snapshot(wl, samples)
    _run(hd, wl)
    _check_tokens_against_oracle(orc, wl, snap, samples)
    wl.ctx.close()
