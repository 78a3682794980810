"""Seeded synthetic inputs for hybrid sliding/full GQA decode attention.

This module only draws numbers: it holds none of the attention arithmetic and
imports neither the CUDA library nor the oracle, so both sides can take their
inputs from it.  Host inputs come from numpy's PCG64 (stable across machines
and versions) and are rounded to bf16 by torch's own cast; device-resident
inputs for the large workloads come from a seeded torch CUDA generator.

The workloads mirror the decode step of vllm_omni/edge/spark_export.py
(Spark-X2.5: 28 layers, three sliding-window layers then one full layer,
8 query / 2 kv heads, head_dim 256, window 512 counting the current token,
sliding RoPE 256 dims at theta 1e4, full RoPE 64 dims at theta 5e6).  Caches
are filled with random already-rotated keys, as that page's ``example_inputs``
fills its random caches; unwritten cache entries are NaN so that any read of
one shows up in the output.
"""
from __future__ import annotations

import math

import numpy as np
import torch

SLIDING, FULL = 0, 1
LAYOUT_AUTO, LAYOUT_RING, LAYOUT_ROLL = 0, 1, 2
SPARK_LAYER_TYPES = [SLIDING, SLIDING, SLIDING, FULL] * 7
WINDOW = 512
HEAD_DIM = 256
ROPE = {SLIDING: (256, 1.0e4), FULL: (64, 5.0e6)}  # layer type -> (rotary_dim, theta)

# Named workloads.  `lengths` is a recipe, resolved by `context_lengths`.
WORKLOADS = {
    # 1 sliding + 1 full layer, two runs at contexts 64 and 700 (700 wraps the ring).
    "tiny_pair": dict(layer_types=[SLIDING, FULL], batch=2, num_q_heads=8, num_kv_heads=2,
                      lengths=("each", (64, 700)), sink=("normal", 1.0, 0.0)),
    # The 28-layer step at batch 1, context 4096, no sink.
    "step28_b1_c4096": dict(layer_types=SPARK_LAYER_TYPES, batch=1, num_q_heads=8,
                            num_kv_heads=2, lengths=("fixed", 4096), sink=None),
    # The 28-layer step at batch 64, per-sequence contexts uniform in [512, 32768].
    "step28_b64_c512_32768": dict(layer_types=SPARK_LAYER_TYPES, batch=64, num_q_heads=8,
                                  num_kv_heads=2, lengths=("uniform", 512, 32768),
                                  sink=("normal", 1.0, 0.0)),
    # Seven full layers only, batch 4 at context 131072.
    "full7_b4_c131072": dict(layer_types=[FULL] * 7, batch=4, num_q_heads=8, num_kv_heads=2,
                             lengths=("fixed", 131072), sink=("normal", 1.0, 0.0)),
    # A small block for profiler captures: [S,S,S,F], batch 16, same length mix
    # (about 1 GB of full-layer cache: larger than L2, a few GB on the device).
    "block4_b16_c512_32768": dict(layer_types=[SLIDING, SLIDING, SLIDING, FULL], batch=16,
                                  num_q_heads=8, num_kv_heads=2, lengths=("uniform", 512, 32768),
                                  sink=("normal", 1.0, 0.0)),
    # Four sliding layers at batch 64 (268 MB of ring caches): profiler captures of
    # the sliding-layer kernel at the batch of the 28-layer step.
    "sliding4_b64_c512_32768": dict(layer_types=[SLIDING] * 4, batch=64, num_q_heads=8,
                                    num_kv_heads=2, lengths=("uniform", 512, 32768),
                                    sink=("normal", 1.0, 0.0)),
    # Group 8: batch 256, 90% at 8192 and 10% (26 of 256) uniform in [1, 512];
    # sink N(0, variance 2) with a quarter of the heads at -inf.
    "step28_b256_g8_mixed": dict(layer_types=SPARK_LAYER_TYPES, batch=256, num_q_heads=16,
                                 num_kv_heads=2, lengths=("mixed", 8192, 0.10, 512),
                                 sink=("normal", math.sqrt(2.0), 0.25)),
}


def generator(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> torch.Tensor:
    """N(0, std^2) samples drawn in fp32 and cast to bf16 by torch (CPU tensor)."""
    x = rng.standard_normal(size=tuple(shape), dtype=np.float32)
    if std != 1.0:
        x = x * np.float32(std)
    return torch.from_numpy(x).to(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor, or the uint8 codes of an E4M3 cache
    (a copy on the host)."""
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return t.view(torch.uint8).numpy().copy()
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def from_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def context_lengths(rng: np.random.Generator, recipe, batch: int) -> np.ndarray:
    """Per-sequence number of previous tokens c_b (int32)."""
    kind = recipe[0]
    if kind == "fixed":
        return np.full(batch, recipe[1], np.int32)
    if kind == "uniform":
        return rng.integers(recipe[1], recipe[2] + 1, size=batch).astype(np.int32)
    if kind == "mixed":
        long_ctx, frac_short, short_max = recipe[1:]
        n_short = int(round(frac_short * batch))
        ctx = np.full(batch, long_ctx, np.int32)
        idx = rng.choice(batch, size=n_short, replace=False)
        ctx[idx] = rng.integers(1, short_max + 1, size=n_short)
        return ctx
    raise ValueError(f"unknown length recipe {recipe!r}")


def sink_vector(rng: np.random.Generator, recipe, num_q_heads: int):
    """Per-head fp32 sink, or None.  recipe = ("normal", std, fraction at -inf)."""
    if recipe is None:
        return None
    _, std, frac_neg_inf = recipe
    s = (rng.standard_normal(num_q_heads) * std).astype(np.float32)
    k = int(math.floor(frac_neg_inf * num_q_heads))
    if k:
        s[rng.choice(num_q_heads, size=k, replace=False)] = -np.inf
    return torch.from_numpy(s)


def gate_logits(rng: np.random.Generator, batch: int, num_q_heads: int, std: float = 1.0,
                specials: bool = False):
    """fp32 [batch][num_q_heads] output-gate logits N(0, std^2); with ``specials``
    the first sequence's heads cycle through +inf, -inf, 0, 30 and -30."""
    g = (rng.standard_normal((batch, num_q_heads)) * std).astype(np.float32)
    if specials:
        vals = np.array([np.inf, -np.inf, 0.0, 30.0, -30.0], np.float32)
        g[0] = vals[np.arange(num_q_heads) % len(vals)]
    return torch.from_numpy(g)


def cache_with_history(rng: np.random.Generator, batch: int, num_kv_heads: int, capacity: int,
                       written, head_dim: int = HEAD_DIM) -> torch.Tensor:
    """bf16 cache [B, Hkv, capacity, D]: entries [0, written[b]) random N(0,1), the rest NaN."""
    t = normal_bf16(rng, (batch, num_kv_heads, capacity, head_dim))
    for b in range(batch):
        t[b, :, int(written[b]):, :] = float("nan")
    return t


E4M3_NAN = 0x7F


def kv_scales(rng: np.random.Generator, num_kv_heads: int) -> torch.Tensor:
    """Per-kv-head fp32 scales amax / 448 for E4M3 caches, amax ~ U[3, 6] (an N(0,1)
    cache spans about +-4.5, so the largest entries sometimes saturate)."""
    return torch.from_numpy((rng.uniform(3.0, 6.0, num_kv_heads) / 448.0).astype(np.float32))


def e4m3_codes(x: torch.Tensor) -> torch.Tensor:
    """uint8 E4M3 codes of a float tensor: torch's float8_e4m3fn cast after clamping
    to the largest finite value (the cast itself maps overflow to NaN)."""
    return x.float().clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def cache_with_history_fp8(rng: np.random.Generator, batch: int, num_kv_heads: int, capacity: int,
                           written, scale: torch.Tensor, head_dim: int = HEAD_DIM) -> torch.Tensor:
    """E4M3 cache [B, Hkv, capacity, D] (uint8 codes): entries [0, written[b]) hold the
    codes of N(0,1) / scale[h], the rest the NaN code."""
    x = rng.standard_normal(size=(batch, num_kv_heads, capacity, head_dim), dtype=np.float32)
    x = x / scale.numpy()[None, :, None, None]
    c = e4m3_codes(torch.from_numpy(x))
    for b in range(batch):
        c[b, :, int(written[b]):, :] = E4M3_NAN
    return c


def cuda_e4m3_codes_(t: torch.Tensor, scale: torch.Tensor, seed: int) -> torch.Tensor:
    """Fill a CUDA uint8 cache [B, Hkv, cap, D] in place with the E4M3 codes of
    seeded N(0,1) / scale[h] samples (one sequence and head at a time)."""
    g = torch.Generator(device=t.device)
    g.manual_seed(seed)
    for b in range(t.shape[0]):
        for h in range(t.shape[1]):
            x = torch.randn(t.shape[2:], generator=g, device=t.device, dtype=torch.float32)
            t[b, h].copy_(e4m3_codes(x / scale[h]))
    return t


def cuda_normal_bf16_(t: torch.Tensor, seed: int) -> torch.Tensor:
    """Fill a CUDA bf16 tensor in place with seeded N(0,1) samples (chunked)."""
    g = torch.Generator(device=t.device)
    g.manual_seed(seed)
    flat = t.view(-1)
    step = 1 << 28
    for i in range(0, flat.numel(), step):
        n = min(step, flat.numel() - i)
        flat[i:i + n] = torch.randn(n, generator=g, device=t.device, dtype=torch.float32).to(t.dtype)
    return t
