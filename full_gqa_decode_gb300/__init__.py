"""Python binding of the hybrid decode-attention C ABI (include/hybrid_decode.h).

Argument marshalling only: every step of the path runs in the CUDA kernels of
``libhybriddecode.so``.  PyTorch provides device memory and streams; tensors
are passed as raw device pointers.  Importing this package loads the in-tree
library and raises if it has not been built -- there is no fallback.

Names follow the C entry points: ``hybrid_decode_init``, ``rope_append_kv``,
``decode_attn_sliding``, ``decode_attn_full``, ``decode_step`` (plus
``hybrid_decode_destroy`` and the helpers).  Each call raises ``HDError``
carrying the hd_status when the library rejects it.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(PKG, "libhybriddecode.so")

HD_SLIDING, HD_FULL = 0, 1
HD_LAYOUT_AUTO, HD_LAYOUT_RING, HD_LAYOUT_ROLL = 0, 1, 2
HD_CONSUMER_CUDA_CORE, HD_CONSUMER_TENSOR_CORE, HD_CONSUMER_TENSOR_MEMORY = 0, 1, 2
HD_PROFILE_SLIDING, HD_PROFILE_FULL, HD_PROFILE_FIRST_ONLY, HD_PROFILE_STEP = 1 << HD_SLIDING, 1 << HD_FULL, 4, 8
HD_PROFILE_KIND_STEP = 2
HD_KV_BF16, HD_KV_FP8_E4M3 = 0, 1
HD_STATIC_SCRATCH_BYTES = 64 << 20   # the allocation-free entry point's scratch array
STATUS = {0: "HD_OK", 1: "HD_ERR_INVALID_ARG", 2: "HD_ERR_UNSUPPORTED", 3: "HD_ERR_CAPACITY",
          4: "HD_ERR_CUDA", 5: "HD_ERR_STATE"}
DEVERR = {1: "HD_DEVERR_CONTEXT_NEGATIVE", 2: "HD_DEVERR_CONTEXT_CAPACITY",
          4: "HD_DEVERR_CONTEXT_PLAN", 8: "HD_DEVERR_WAIT_TIMEOUT"}

if not os.path.exists(LIBRARY):
    raise ImportError(f"{LIBRARY} is missing: build it with full_gqa_decode_gb300.build.build() "
                      "(or __graft_entry__.build()); there is no non-CUDA fallback")
_lib = ctypes.CDLL(LIBRARY)


class HDError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class hd_config(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("layer_types", ctypes.POINTER(ctypes.c_int32)),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("sliding_window", ctypes.c_int32),
                ("rotary_dim_sliding", ctypes.c_int32), ("rotary_dim_full", ctypes.c_int32),
                ("rope_theta_sliding", ctypes.c_double), ("rope_theta_full", ctypes.c_double),
                ("cache_layout", ctypes.c_int32), ("max_batch", ctypes.c_int32),
                ("max_context", ctypes.c_int32), ("kv_dtype", ctypes.c_int32)]


class hd_kv_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("seq_stride", ctypes.c_int64),
                ("capacity", ctypes.c_int32), ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p)]


class hd_layer_io(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("cache", hd_kv_cache), ("sink", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("lse", ctypes.c_void_p), ("gate", ctypes.c_void_p)]


_c = ctypes
_P = _c.c_void_p
_i32, _i64 = _c.c_int32, _c.c_int64
_SIGS = {
    "hd_validate_config": [_c.POINTER(hd_config)],
    "hd_plan_split": [_i32, _i32, _i32, _i32, _c.POINTER(_i32), _c.POINTER(_i32)],
    "hd_plan_step_split": [_i32, _c.POINTER(_i32), _c.POINTER(_c.c_uint8), _i32, _i32, _i32, _i32, _i32, _i32,
                           _c.POINTER(_i32)],
    "hybrid_decode_init": [_c.POINTER(hd_config), _c.POINTER(_P)],
    "hybrid_decode_destroy": [_P],
    "rope_append_kv": [_P, _i32, _i32, _P, _P, _P, _P, _P, hd_kv_cache, _P],
    "decode_attn_sliding": [_P, _i32, _i32, _P, _P, hd_kv_cache, _P, _P, _P, _P, _P],
    "decode_attn_full": [_P, _i32, _i32, _P, _i32, _P, hd_kv_cache, _P, _P, _P, _P, _P],
    "decode_step": [_P, _i32, _P, _i32, _c.POINTER(hd_layer_io), _P],
    "decode_step_tokens": [_P, _i32, _i32, _P, _i32, _c.POINTER(hd_layer_io), _P],
    "hybrid_decode_device_errors": [_P, _c.POINTER(_i32), _P],
    "hybrid_decode_launch_count": [_P, _c.POINTER(_i64)],
    "hybrid_decode_set_profiling": [_P, _i32],
    "hybrid_decode_profile": [_P, _i32, _c.POINTER(_c.c_double), _c.POINTER(_i64)],
    "hybrid_decode_set_consumer": [_P, _i32],
    "decode_attn_full_static_scratch": [_i32, _i32, _i32, _P, _i32, _P, hd_kv_cache, _P, _P, _P, _P],
    "decode_attn_full_static_scratch_plan": [_i32, _i32, _i32, _i32, _i32, _c.POINTER(_i64), _c.POINTER(_i32),
                                             _c.POINTER(_i32)],
    "hybrid_decode_read_probe": [_P, _i64, _P],
    "hybrid_decode_inject_lost_copy": [_P, _i32],
    "hybrid_decode_set_layer_overlap": [_P, _i32],
    "hybrid_decode_set_step_fusion": [_P, _i32],
    "hybrid_decode_set_cluster_combine": [_P, _i32],
}
for _name, _args in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _c.c_int
_lib.hd_status_string.argtypes = [_c.c_int]
_lib.hd_status_string.restype = _c.c_char_p


def _check(status: int, what: str) -> None:
    if status != 0:
        raise HDError(status, what)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _check_sink(sink, num_q_heads: int, like: torch.Tensor) -> None:
    """Sink checks of vllm/models/hy_v4/nvidia/flashmla_sparse.py (`_validate_sinks`,
    `_sinks_for_query`): fp32, shape (num_q_heads,), on the query's device."""
    if sink is None:
        return
    if sink.dtype != torch.float32:
        raise ValueError(f"sink must be float32, got {sink.dtype}")
    if sink.dim() != 1 or sink.shape[0] != num_q_heads:
        raise ValueError(f"sink must have shape ({num_q_heads},), got {tuple(sink.shape)}")
    if sink.device != like.device:
        raise ValueError(f"sink and query must be on the same device ({sink.device} vs {like.device})")
    if not sink.is_contiguous():
        raise ValueError("sink must be contiguous")


def _check_gate(gate, batch: int, num_q_heads: int, like: torch.Tensor, tokens: int | None = None) -> None:
    """Output-gate logits: fp32, shape (batch, num_q_heads) -- or (batch, tokens,
    num_q_heads) for a multi-token step -- contiguous, on the query's device."""
    if gate is None:
        return
    if gate.dtype != torch.float32:
        raise ValueError(f"gate must be float32, got {gate.dtype}")
    want = (batch, num_q_heads) if tokens is None else (batch, tokens, num_q_heads)
    if tuple(gate.shape) != want:
        raise ValueError(f"gate must have shape {want}, got {tuple(gate.shape)}")
    if gate.device != like.device:
        raise ValueError(f"gate and query must be on the same device ({gate.device} vs {like.device})")
    if not gate.is_contiguous():
        raise ValueError("gate must be contiguous")


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


@dataclass
class Config:
    """Model shape; field meanings follow ``hd_config`` in include/hybrid_decode.h."""
    layer_types: list
    num_q_heads: int = 8
    num_kv_heads: int = 2
    head_dim: int = 256
    sliding_window: int = 512
    rotary_dim_sliding: int = 256
    rotary_dim_full: int = 64
    rope_theta_sliding: float = 1.0e4
    rope_theta_full: float = 5.0e6
    cache_layout: int = HD_LAYOUT_AUTO
    max_batch: int = 1
    max_context: int = 4096
    kv_dtype: int = HD_KV_BF16
    _types: object = field(default=None, repr=False)

    def to_c(self) -> hd_config:
        self._types = (ctypes.c_int32 * len(self.layer_types))(*self.layer_types)
        return hd_config(len(self.layer_types), self._types, self.num_q_heads, self.num_kv_heads,
                         self.head_dim, self.sliding_window, self.rotary_dim_sliding,
                         self.rotary_dim_full, self.rope_theta_sliding, self.rope_theta_full,
                         self.cache_layout, self.max_batch, self.max_context, self.kv_dtype)


_FP8_CACHE_TYPES = (torch.uint8, torch.float8_e4m3fn)


def kv_cache(k: torch.Tensor, v: torch.Tensor, k_scale: torch.Tensor | None = None,
             v_scale: torch.Tensor | None = None) -> hd_kv_cache:
    """Describe a cache pair shaped [batch, num_kv_heads, capacity, head_dim] on CUDA:
    bf16, or E4M3 codes (uint8 or float8_e4m3fn) with fp32 ``k_scale``/``v_scale``
    of shape [num_kv_heads] on the same device (the context's kv_dtype must match)."""
    if k.shape != v.shape or k.dim() != 4 or k.stride() != v.stride():
        raise ValueError("k and v caches must share a [batch, kv_heads, capacity, head_dim] layout")
    fp8 = k.dtype in _FP8_CACHE_TYPES
    if fp8:
        if v.dtype not in _FP8_CACHE_TYPES:
            raise ValueError("k and v caches must have the same element type")
        for name, sc in (("k_scale", k_scale), ("v_scale", v_scale)):
            if sc is None or sc.dtype != torch.float32 or tuple(sc.shape) != (k.shape[1],):
                raise ValueError(f"an FP8 cache needs {name} as float32 of shape ({k.shape[1]},)")
            if sc.device != k.device or not sc.is_contiguous():
                raise ValueError(f"{name} must be contiguous and on the cache's device")
    else:
        if k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
            raise ValueError("caches must be bf16, or E4M3 codes with scales")
        if k_scale is not None or v_scale is not None:
            raise ValueError("scales belong to FP8 caches only")
    if k.stride(3) != 1 or k.stride(2) != k.shape[3] or k.stride(1) != k.shape[2] * k.shape[3]:
        raise ValueError("each sequence's cache must be contiguous [kv_heads, capacity, head_dim]")
    if not k.is_cuda or not v.is_cuda:
        raise ValueError("caches must be CUDA tensors")
    c = hd_kv_cache(k.data_ptr(), v.data_ptr(), k.stride(0), k.shape[2],
                    k_scale.data_ptr() if fp8 else None, v_scale.data_ptr() if fp8 else None)
    c.batch = k.shape[0]  # sequences the tensors hold; calls may not pass a larger batch
    c.keep = (k_scale, v_scale)  # the scales must outlive the descriptor
    return c


def _check_batch(cache: hd_kv_cache, batch: int) -> None:
    held = getattr(cache, "batch", None)
    if held is not None and held < batch:
        raise ValueError(f"cache holds {held} sequences, call passes batch {batch}")


def hd_validate_config(cfg: Config) -> int:
    return _lib.hd_validate_config(ctypes.byref(cfg.to_c()))


def hd_plan_split(batch: int, num_kv_heads: int, max_keys: int, num_sms: int) -> tuple[int, int]:
    ck, nc = ctypes.c_int32(), ctypes.c_int32()
    _check(_lib.hd_plan_split(batch, num_kv_heads, max_keys, num_sms, ctypes.byref(ck),
                              ctypes.byref(nc)), "hd_plan_split")
    return ck.value, nc.value


def hd_plan_step_split(max_keys, batch: int, num_kv_heads: int, rows: int, num_sms: int,
                       kv_dtype: int = 0, multi_token: bool = False, one_chunk=None) -> int:
    """Chunk size decode_step's step grid uses for layers scoring at most max_keys[i] keys."""
    n = len(max_keys)
    mk = (ctypes.c_int32 * n)(*[int(x) for x in max_keys])
    oc = None if one_chunk is None else (ctypes.c_uint8 * n)(*[1 if x else 0 for x in one_chunk])
    ck = ctypes.c_int32()
    _check(_lib.hd_plan_step_split(n, mk, oc, batch, num_kv_heads, rows, int(bool(multi_token)), kv_dtype,
                                   num_sms, ctypes.byref(ck)), "hd_plan_step_split")
    return ck.value


def hd_status_string(status: int) -> str:
    return _lib.hd_status_string(status).decode()


class Context:
    """Owns one ``hd_ctx``; create it with ``hybrid_decode_init``."""

    def __init__(self, handle: int, cfg: Config):
        self.handle = handle
        self.cfg = cfg

    def close(self) -> None:
        if self.handle:
            _check(_lib.hybrid_decode_destroy(self.handle), "hybrid_decode_destroy")
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def hybrid_decode_init(cfg: Config) -> Context:
    h = ctypes.c_void_p()
    _check(_lib.hybrid_decode_init(ctypes.byref(cfg.to_c()), ctypes.byref(h)), "hybrid_decode_init")
    return Context(h.value, cfg)


def hybrid_decode_destroy(ctx: Context) -> None:
    ctx.close()


def rope_append_kv(ctx: Context, layer: int, context: torch.Tensor, q, k, v, q_rot, cache: hd_kv_cache,
                   stream=None) -> None:
    _check_batch(cache, q.shape[0])
    _check(_lib.rope_append_kv(ctx.handle, layer, q.shape[0], _ptr(context), _ptr(q), _ptr(k), _ptr(v),
                               _ptr(q_rot), cache, _stream(stream)), "rope_append_kv")


def decode_attn_sliding(ctx: Context, layer: int, context, q_rot, cache: hd_kv_cache, sink, out, lse,
                        stream=None, gate=None) -> None:
    _check_sink(sink, ctx.cfg.num_q_heads, q_rot)
    _check_gate(gate, q_rot.shape[0], ctx.cfg.num_q_heads, q_rot)
    _check_batch(cache, q_rot.shape[0])
    _check(_lib.decode_attn_sliding(ctx.handle, layer, q_rot.shape[0], _ptr(context), _ptr(q_rot),
                                    cache, _ptr(sink), _ptr(gate), _ptr(out), _ptr(lse), _stream(stream)),
           "decode_attn_sliding")


def decode_attn_full(ctx: Context, layer: int, context, q_rot, cache: hd_kv_cache, sink, out, lse,
                     max_context_hint: int = 0, stream=None, gate=None) -> None:
    _check_sink(sink, ctx.cfg.num_q_heads, q_rot)
    _check_gate(gate, q_rot.shape[0], ctx.cfg.num_q_heads, q_rot)
    _check_batch(cache, q_rot.shape[0])
    _check(_lib.decode_attn_full(ctx.handle, layer, q_rot.shape[0], _ptr(context), max_context_hint,
                                 _ptr(q_rot), cache, _ptr(sink), _ptr(gate), _ptr(out), _ptr(lse),
                                 _stream(stream)), "decode_attn_full")


def layer_io(q, k, v, cache: hd_kv_cache, sink, out, lse, gate=None) -> hd_layer_io:
    """One layer's tensors for decode_step (q [B, Hq, D]) or decode_step_tokens
    (q [B, T, Hq, D]; k/v/out/lse/gate with the same token index)."""
    if sink is not None:
        _check_sink(sink, q.shape[-2], q)
    _check_gate(gate, q.shape[0], q.shape[-2], q, tokens=q.shape[1] if q.dim() == 4 else None)
    _check_batch(cache, q.shape[0])
    return hd_layer_io(_ptr(q), _ptr(k), _ptr(v), cache, _ptr(sink), _ptr(out), _ptr(lse), _ptr(gate))


def layer_array(ctx: Context, layers) -> ctypes.Array:
    """The host array of hd_layer_io decode_step reads, one entry per layer of the
    context; build it once and pass it to every step whose tensors stay the same."""
    if isinstance(layers, ctypes.Array) and layers._type_ is hd_layer_io:
        arr = layers
    else:
        arr = (hd_layer_io * len(layers))(*layers)
    if len(arr) != len(ctx.cfg.layer_types):
        raise ValueError(f"decode_step needs one hd_layer_io per layer ({len(ctx.cfg.layer_types)}), got {len(arr)}")
    return arr


def decode_step(ctx: Context, context: torch.Tensor, layers, batch: int,
                max_context_hint: int = 0, stream=None) -> None:
    """layers: a list of hd_layer_io (one per layer) or an array from layer_array()."""
    _check(_lib.decode_step(ctx.handle, batch, _ptr(context), max_context_hint, layer_array(ctx, layers),
                            _stream(stream)), "decode_step")


def decode_step_tokens(ctx: Context, context: torch.Tensor, layers: list, batch: int, num_tokens: int,
                       max_context_hint: int = 0, stream=None) -> None:
    """num_tokens new tokens per sequence (q/out [B, T, Hq, D], k/v [B, T, Hkv, D],
    lse/gate [B, T, Hq]), equal to num_tokens decode_step calls in order.  layers as
    for decode_step."""
    _check(_lib.decode_step_tokens(ctx.handle, batch, num_tokens, _ptr(context), max_context_hint,
                                   layer_array(ctx, layers), _stream(stream)), "decode_step_tokens")


def hybrid_decode_device_errors(ctx: Context, stream=None) -> int:
    f = ctypes.c_int32()
    _check(_lib.hybrid_decode_device_errors(ctx.handle, ctypes.byref(f), _stream(stream)),
           "hybrid_decode_device_errors")
    return f.value


def hybrid_decode_launch_count(ctx: Context) -> int:
    n = ctypes.c_int64()
    _check(_lib.hybrid_decode_launch_count(ctx.handle, ctypes.byref(n)), "hybrid_decode_launch_count")
    return n.value


def hybrid_decode_set_profiling(ctx: Context, mask: int) -> None:
    """mask of launches to bracket with events: HD_PROFILE_SLIDING | HD_PROFILE_FULL (layer
    kernels), HD_PROFILE_STEP (step grids), or 0; with HD_PROFILE_FIRST_ONLY only the first
    layer kernel of each type per decode_step."""
    _check(_lib.hybrid_decode_set_profiling(ctx.handle, int(mask)), "hybrid_decode_set_profiling")


def hybrid_decode_profile(ctx: Context, layer_type: int = HD_FULL) -> tuple[float, int]:
    """(summed kernel milliseconds, launches) of the given layer type (or HD_PROFILE_KIND_STEP:
    step grids) since the last read."""
    ms, n = ctypes.c_double(), ctypes.c_int64()
    _check(_lib.hybrid_decode_profile(ctx.handle, layer_type, ctypes.byref(ms), ctypes.byref(n)),
           "hybrid_decode_profile")
    return ms.value, n.value


def hybrid_decode_set_layer_overlap(ctx: Context, enable: bool) -> None:
    """Whether decode_step lets a layer start before the previous one finishes (default on)."""
    _check(_lib.hybrid_decode_set_layer_overlap(ctx.handle, int(bool(enable))), "hybrid_decode_set_layer_overlap")


def hybrid_decode_set_step_fusion(ctx: Context, enable: bool) -> None:
    """Whether decode_step runs the attention of all layers as one grid (default on)."""
    _check(_lib.hybrid_decode_set_step_fusion(ctx.handle, int(bool(enable))), "hybrid_decode_set_step_fusion")


def hybrid_decode_set_cluster_combine(ctx: Context, enable: bool) -> None:
    """Single-layer launches of small grids merge their chunks inside a
    thread-block cluster (default True), or through the workspace (False)."""
    _check(_lib.hybrid_decode_set_cluster_combine(ctx.handle, 1 if enable else 0), "hybrid_decode_set_cluster_combine")


def hybrid_decode_set_consumer(ctx: Context, consumer: int) -> None:
    """HD_CONSUMER_CUDA_CORE, HD_CONSUMER_TENSOR_CORE (the default) or
    HD_CONSUMER_TENSOR_MEMORY (tcgen05 for 16-row multi-token passes over bf16 caches)."""
    _check(_lib.hybrid_decode_set_consumer(ctx.handle, consumer), "hybrid_decode_set_consumer")


def decode_attn_full_static_scratch(num_kv_heads: int, context, max_context: int, q_rot,
                                    cache: hd_kv_cache, sink, out, lse, stream=None) -> None:
    """Full-layer attention without a context and without any allocation: for
    callers that cannot allocate device memory while running.  The scratch is a
    64 MiB array inside the library, shared by all calls: calls that overlap on
    the GPU race, so order them on one stream.  See include/hybrid_decode.h."""
    batch, num_q_heads = q_rot.shape[0], q_rot.shape[1]
    _check_sink(sink, num_q_heads, q_rot)
    _check_batch(cache, batch)
    _check(_lib.decode_attn_full_static_scratch(batch, num_q_heads, num_kv_heads, _ptr(context),
                                                max_context, _ptr(q_rot), cache, _ptr(sink), _ptr(out),
                                                _ptr(lse), _stream(stream)),
           "decode_attn_full_static_scratch")


def decode_attn_full_static_scratch_plan(batch: int, num_q_heads: int, num_kv_heads: int, max_context: int,
                                         num_sms: int) -> tuple[int, int, int, int]:
    """(scratch bytes, keys per chunk, chunks, status) of decode_attn_full_static_scratch
    for this shape (pure host function).  Status 0: the call fits the array; 3
    (HD_ERR_CAPACITY): it would be refused; 1 / 2: the shape is rejected."""
    nbytes, chunk, chunks = _i64(0), _i32(0), _i32(0)
    st = _lib.decode_attn_full_static_scratch_plan(batch, num_q_heads, num_kv_heads, max_context, num_sms,
                                                   ctypes.byref(nbytes), ctypes.byref(chunk), ctypes.byref(chunks))
    return nbytes.value, chunk.value, chunks.value, st


def hybrid_decode_read_probe(buffer: torch.Tensor, stream=None) -> int:
    """One pass of a pure read stream over a device buffer; returns the bytes the
    pass covers (a whole number of 32 KiB stages per CTA).  Time it with events."""
    nbytes = buffer.numel() * buffer.element_size()
    _check(_lib.hybrid_decode_read_probe(_ptr(buffer), nbytes, _stream(stream)), "hybrid_decode_read_probe")
    ctas = 2 * torch.cuda.get_device_properties(buffer.device).multi_processor_count
    return (nbytes // (32 * 1024) // ctas) * ctas * 32 * 1024


def hybrid_decode_inject_lost_copy(ctx: Context, stage: int) -> None:
    """Test hook: attention producers stop issuing copies at `stage` (-1: off)."""
    _check(_lib.hybrid_decode_inject_lost_copy(ctx.handle, stage), "hybrid_decode_inject_lost_copy")
