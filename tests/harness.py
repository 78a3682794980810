"""Shared helpers of the GPU parity tests: run one layer through the C ABI and
through the oracle on the same seeded inputs, and compare.

Tolerances (written here, used by every parity test):
  out  |gpu - ref| <= OUT_ATOL + OUT_RTOL * |ref|  elementwise (bf16 output,
       fp32 accumulation; the abs 1e-2 / rel 1e-2 bound in allclose form)
  lse  |gpu - ref| <= LSE_ATOL
  written K/V, slot indices, untouched cache entries: bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import synth

OUT_ATOL = 1e-2
OUT_RTOL = 1e-2
LSE_ATOL = 1e-3
SLIDING, FULL = synth.SLIDING, synth.FULL
RING, ROLL = synth.LAYOUT_RING, synth.LAYOUT_ROLL


def assert_out_close(gpu_out: torch.Tensor, ref: np.ndarray, what: str = "out") -> float:
    g = gpu_out.detach().float().cpu().double().numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    excess = np.abs(g - ref) - (OUT_ATOL + OUT_RTOL * np.abs(ref))
    worst = float(excess.max())
    assert worst <= 0.0, f"{what}: max excess over tolerance {worst:.3e} at {np.unravel_index(excess.argmax(), excess.shape)}"
    return float(np.abs(g - ref).max())


def assert_lse_close(gpu_lse: torch.Tensor, ref: np.ndarray, what: str = "lse") -> float:
    g = gpu_lse.detach().cpu().double().numpy()
    d = np.abs(g - ref)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU lse"
    assert d.max() <= LSE_ATOL, f"{what}: max |dlse| = {d.max():.3e}"
    return float(d.max())


def assert_bits_equal(gpu: torch.Tensor, ref_bits: np.ndarray, what: str) -> None:
    g = synth.bits(gpu)
    if not np.array_equal(g, ref_bits):
        idx = np.argwhere(g != ref_bits)
        raise AssertionError(f"{what}: {len(idx)} entries differ, first at {tuple(idx[0])}")


class LayerCase:
    """Seeded inputs of one layer call: q/k/v, caches with `written` valid entries
    (bf16, or E4M3 codes with per-kv-head scales when kv == "fp8")."""

    def __init__(self, rng, batch, num_q_heads, num_kv_heads, capacity, context, written=None,
                 sink=None, gate=None, kv="bf16", k_std=1.0):
        D = synth.HEAD_DIM
        self.context = np.asarray(context, np.int32)
        self.q = synth.normal_bf16(rng, (batch, num_q_heads, D))
        self.k = synth.normal_bf16(rng, (batch, num_kv_heads, D), std=k_std)
        self.v = synth.normal_bf16(rng, (batch, num_kv_heads, D), std=k_std)
        if written is None:
            written = np.minimum(self.context, capacity)
        self.kv = kv
        self.k_scale = self.v_scale = None
        if kv == "fp8":
            self.k_scale = synth.kv_scales(rng, num_kv_heads)
            self.v_scale = synth.kv_scales(rng, num_kv_heads)
            self.kc = synth.cache_with_history_fp8(rng, batch, num_kv_heads, capacity, written, self.k_scale, D)
            self.vc = synth.cache_with_history_fp8(rng, batch, num_kv_heads, capacity, written, self.v_scale, D)
        else:
            self.kc = synth.cache_with_history(rng, batch, num_kv_heads, capacity, written, D)
            self.vc = synth.cache_with_history(rng, batch, num_kv_heads, capacity, written, D)
        self.sink = sink
        self.gate = gate  # fp32 [batch][num_q_heads] output-gate logits, or None

    def cache(self, hd, kd, vd, dev):
        if self.kv == "fp8":
            # the descriptor holds raw pointers: keep the device scales alive with the case
            self.scales_dev = (self.k_scale.to(dev), self.v_scale.to(dev))
            return hd.kv_cache(kd, vd, *self.scales_dev)
        return hd.kv_cache(kd, vd)


def oracle_layer(orc, case: LayerCase, layer_type: int, layout: int, rotary_dim=None, theta=None):
    rot, th = synth.ROPE[layer_type]
    kc, vc = synth.bits(case.kc), synth.bits(case.vc)
    r = orc.decode_layer(layer_type=layer_type, layout=layout if layer_type == SLIDING else 0,
                         window=synth.WINDOW, rotary_dim=rotary_dim or rot, rope_theta=theta or th,
                         context=case.context, q=synth.bits(case.q), k=synth.bits(case.k),
                         v=synth.bits(case.v), kcache=kc, vcache=vc,
                         sink=None if case.sink is None else case.sink.numpy(),
                         gate=None if case.gate is None else case.gate.numpy(),
                         k_scale=None if case.k_scale is None else case.k_scale.numpy(),
                         v_scale=None if case.v_scale is None else case.v_scale.numpy())
    r["kcache"], r["vcache"] = kc, vc
    return r


def gpu_layer(hd, ctx, layer: int, layer_type: int, case: LayerCase, max_context_hint: int = 0):
    dev = torch.device("cuda")
    B, Hq, D = case.q.shape
    ctx_d = torch.from_numpy(case.context).to(dev)
    kd, vd = case.kc.to(dev), case.vc.to(dev)
    qrot = torch.empty(B, Hq, D, dtype=torch.float32, device=dev)
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    cache = case.cache(hd, kd, vd, dev)
    sink = None if case.sink is None else case.sink.to(dev)
    gate = None if case.gate is None else case.gate.to(dev)
    hd.rope_append_kv(ctx, layer, ctx_d, case.q.to(dev), case.k.to(dev), case.v.to(dev), qrot, cache)
    if layer_type == SLIDING:
        hd.decode_attn_sliding(ctx, layer, ctx_d, qrot, cache, sink, out, lse, gate=gate)
    else:
        hd.decode_attn_full(ctx, layer, ctx_d, qrot, cache, sink, out, lse,
                            max_context_hint=max_context_hint, gate=gate)
    torch.cuda.synchronize()
    flags = hd.hybrid_decode_device_errors(ctx)
    return {"qrot": qrot, "out": out, "lse": lse, "kcache": kd, "vcache": vd, "flags": flags}


def check_layer(hd, orc, ctx, layer, layer_type, layout, case, max_context_hint=0):
    ref = oracle_layer(orc, case, layer_type, layout)
    got = gpu_layer(hd, ctx, layer, layer_type, case, max_context_hint)
    assert got["flags"] == 0, f"device error flags {got['flags']:#x}"
    q = got["qrot"].cpu().double().numpy()
    assert np.allclose(q, ref["qrot"], rtol=1e-5, atol=1e-5), "q_rot"
    assert_out_close(got["out"], ref["out"])
    assert_lse_close(got["lse"], ref["lse"])
    assert_bits_equal(got["kcache"], ref["kcache"], "K cache after the step")
    assert_bits_equal(got["vcache"], ref["vcache"], "V cache after the step")
    return ref, got
