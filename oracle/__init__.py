"""fp64 CPU oracle for hybrid sliding/full GQA decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this package.  The
product path (``full_gqa_decode_gb300``) never imports, links or runs it, and
this package never imports the product.

The arithmetic lives in ``hd_oracle.c`` (plain C, fp64, single thread per
call); this module only compiles it with gcc and marshals numpy arrays through
ctypes.  bf16 values travel as their uint16 bit patterns.

Sources: vllm_omni/edge/spark_export.py (Spark-X2.5 decode step: ``_angles``,
``_rope``, ``_Layer.forward``, ``cache_len``, ``kv_cache_bytes``) and
vllm/models/hy_v4/nvidia/flashmla_sparse.py (the per-head sink).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "hd_oracle.c")
LIBRARY = os.path.join(HERE, "libhd_oracle.so")

SLIDING, FULL = 0, 1
LAYOUT_RING, LAYOUT_ROLL = 1, 2
KV_BF16, KV_FP8_E4M3 = 0, 1

_u8p = ctypes.POINTER(ctypes.c_uint8)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)


class OrcLayer(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("layer_type", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("window", ctypes.c_int32),
        ("rotary_dim", ctypes.c_int32),
        ("rope_theta", ctypes.c_double),
        ("capacity", ctypes.c_int32),
        ("seq_stride", ctypes.c_int64),
        ("kv_dtype", ctypes.c_int32),
    ]


def build(source: str = SOURCE, output: str = LIBRARY, defines: tuple = ()) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", *[f"-D{d}" for d in defines], source, "-o", output, "-lm"]
    subprocess.run(cmd, check=True)
    return output


_lock = threading.Lock()
_libs: dict[str, "Oracle"] = {}


def _stale(lib: str, src: str) -> bool:
    return not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src)


def load(path: str | None = None) -> "Oracle":
    """Return the oracle bound to ``path`` (default: the in-tree build)."""
    path = path or LIBRARY
    with _lock:
        if path not in _libs:
            if path == LIBRARY and _stale(LIBRARY, SOURCE):
                build()
            _libs[path] = Oracle(path)
        return _libs[path]


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.orc_bf16_to_f64.restype = ctypes.c_double
        lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_f64_to_bf16.restype = ctypes.c_uint16
        lib.orc_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.orc_rope_angles.restype = None
        lib.orc_rope_angles.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_double, _f32p, _f32p]
        lib.orc_rope_f64.restype = None
        lib.orc_rope_f64.argtypes = [_f64p, ctypes.c_int, ctypes.c_int, _f32p, _f32p, _f64p]
        lib.orc_attend.restype = None
        lib.orc_attend.argtypes = [_f64p, ctypes.c_int, ctypes.c_int, _f64p, _f64p,
                                   ctypes.c_int, ctypes.c_double, _f64p, _f64p]
        lib.orc_cache_len.restype = ctypes.c_int64
        lib.orc_cache_len.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64]
        lib.orc_kv_cache_bytes.restype = None
        lib.orc_kv_cache_bytes.argtypes = [ctypes.c_int, _i32p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int64, _i64p, _i64p]
        lib.orc_decode_layer.restype = ctypes.c_int
        lib.orc_e4m3_to_f64.restype = ctypes.c_double
        lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.orc_f64_to_e4m3.restype = ctypes.c_uint8
        lib.orc_f64_to_e4m3.argtypes = [ctypes.c_double]
        lib.orc_decode_layer.argtypes = [ctypes.POINTER(OrcLayer), _i32p, _u16p, _u16p, _u16p,
                                         ctypes.c_void_p, ctypes.c_void_p, _f32p, _f32p, _f32p, _f32p,
                                         _f64p, _f64p, _f64p, ctypes.c_void_p]
        lib.orc_decode_tokens.restype = ctypes.c_int
        lib.orc_decode_tokens.argtypes = [ctypes.POINTER(OrcLayer), ctypes.c_int, _i32p, _u16p, _u16p, _u16p,
                                          ctypes.c_void_p, ctypes.c_void_p, _f32p, _f32p, _f32p, _f32p,
                                          _f64p, _f64p]
        self.lib = lib
        self.path = path

    # -- scalars ------------------------------------------------------------
    def bf16_to_f64(self, bits) -> np.ndarray:
        a = np.asarray(bits, dtype=np.uint16)
        return np.array([self.lib.orc_bf16_to_f64(int(b)) for b in a.ravel()]).reshape(a.shape)

    def f64_to_bf16(self, x) -> np.ndarray:
        a = np.asarray(x, dtype=np.float64)
        return np.array([self.lib.orc_f64_to_bf16(float(v)) for v in a.ravel()],
                        dtype=np.uint16).reshape(a.shape)

    def e4m3_to_f64(self, codes) -> np.ndarray:
        a = np.asarray(codes, dtype=np.uint8)
        return np.array([self.lib.orc_e4m3_to_f64(int(c)) for c in a.ravel()]).reshape(a.shape)

    def f64_to_e4m3(self, x) -> np.ndarray:
        a = np.asarray(x, dtype=np.float64)
        return np.array([self.lib.orc_f64_to_e4m3(float(v)) for v in a.ravel()],
                        dtype=np.uint8).reshape(a.shape)

    # -- rotary -------------------------------------------------------------
    def rope_angles(self, position: int, rotary_dim: int, theta: float):
        c = np.zeros(rotary_dim // 2, np.float32)
        s = np.zeros(rotary_dim // 2, np.float32)
        self.lib.orc_rope_angles(int(position), int(rotary_dim), float(theta),
                                 _ptr(c, _f32p), _ptr(s, _f32p))
        return c, s

    def rope(self, x, rotary_dim: int, cos_half, sin_half) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float64)
        c = np.ascontiguousarray(cos_half, dtype=np.float32)
        s = np.ascontiguousarray(sin_half, dtype=np.float32)
        y = np.zeros_like(x)
        self.lib.orc_rope_f64(_ptr(x, _f64p), x.shape[-1], int(rotary_dim),
                              _ptr(c, _f32p), _ptr(s, _f32p), _ptr(y, _f64p))
        return y

    # -- attention ----------------------------------------------------------
    def attend(self, q, keys, vals, sink: float | None = None):
        q = np.ascontiguousarray(q, dtype=np.float64)
        keys = np.ascontiguousarray(keys, dtype=np.float64).reshape(-1, q.shape[0])
        vals = np.ascontiguousarray(vals, dtype=np.float64).reshape(-1, q.shape[0])
        out = np.zeros(q.shape[0])
        lse = np.zeros(1)
        self.lib.orc_attend(_ptr(q, _f64p), q.shape[0], keys.shape[0], _ptr(keys, _f64p),
                            _ptr(vals, _f64p), int(sink is not None),
                            float(sink) if sink is not None else 0.0,
                            _ptr(out, _f64p), _ptr(lse, _f64p))
        return out, float(lse[0])

    # -- geometry -----------------------------------------------------------
    def cache_len(self, layer_type: int, layout: int, window: int, context: int) -> int:
        return int(self.lib.orc_cache_len(layer_type, layout, window, context))

    def kv_cache_bytes(self, layer_types, sliding_layout: int, window: int,
                       num_kv_heads: int, head_dim: int, context: int,
                       bytes_per_elem: int = 2) -> tuple[int, int]:
        t = np.ascontiguousarray(layer_types, dtype=np.int32)
        hyb = ctypes.c_int64()
        uni = ctypes.c_int64()
        self.lib.orc_kv_cache_bytes(len(t), _ptr(t, _i32p), sliding_layout, window,
                                    num_kv_heads, head_dim, bytes_per_elem, int(context),
                                    ctypes.byref(hyb), ctypes.byref(uni))
        return hyb.value, uni.value

    # -- one layer ----------------------------------------------------------
    def decode_layer(self, *, layer_type: int, layout: int, window: int, rotary_dim: int,
                     rope_theta: float, context, q, k, v, kcache, vcache, sink=None, gate=None,
                     k_scale=None, v_scale=None):
        """One decode step of one layer; kcache/vcache are updated in place.

        q [B,Hq,D] and k/v [B,Hkv,D] are uint16 bf16 bit patterns; the caches
        [B,Hkv,cap,D] are uint16 bf16 bits, or uint8 E4M3 codes with fp32
        ``k_scale``/``v_scale`` [Hkv]; ``context`` is int32 [B]; ``sink``
        float32 [Hq] or None; ``gate`` float32 [B, Hq] output-gate logits or None.
        Returns dict(out [B,Hq,D] f64, lse [B,Hq] f64, qrot [B,Hq,D] f64,
        k_written [B,Hkv,D] in the cache's element type).
        """
        for name, a in (("q", q), ("k", k), ("v", v)):
            if a.dtype != np.uint16 or not a.flags.c_contiguous:
                raise ValueError(f"{name} must be C-contiguous uint16 bf16 bits")
        fp8 = kcache.dtype == np.uint8
        for name, a in (("kcache", kcache), ("vcache", vcache)):
            if a.dtype != (np.uint8 if fp8 else np.uint16) or not a.flags.c_contiguous:
                raise ValueError(f"{name} must be C-contiguous, uint16 bf16 bits or uint8 E4M3 codes")
        if fp8 and (k_scale is None or v_scale is None):
            raise ValueError("an FP8 cache needs k_scale and v_scale")
        B, Hq, D = q.shape
        Hkv = k.shape[1]
        cap = kcache.shape[2]
        ctx = np.ascontiguousarray(context, dtype=np.int32)
        L = OrcLayer(B, Hq, Hkv, D, layer_type, layout, window, rotary_dim, float(rope_theta),
                     cap, Hkv * cap * D, KV_FP8_E4M3 if fp8 else KV_BF16)
        out = np.zeros((B, Hq, D))
        lse = np.zeros((B, Hq))
        qrot = np.zeros((B, Hq, D))
        kw = np.zeros((B, Hkv, D), np.uint8 if fp8 else np.uint16)
        ksc = vsc = None
        if fp8:
            ksc = np.ascontiguousarray(k_scale, dtype=np.float32)
            vsc = np.ascontiguousarray(v_scale, dtype=np.float32)
        sk = None
        if sink is not None:
            sk = np.ascontiguousarray(sink, dtype=np.float32)
        gt = None
        if gate is not None:
            gt = np.ascontiguousarray(gate, dtype=np.float32).reshape(B, Hq)
        rc = self.lib.orc_decode_layer(ctypes.byref(L), _ptr(ctx, _i32p), _ptr(q, _u16p),
                                       _ptr(k, _u16p), _ptr(v, _u16p), kcache.ctypes.data,
                                       vcache.ctypes.data,
                                       _ptr(ksc, _f32p) if ksc is not None else None,
                                       _ptr(vsc, _f32p) if vsc is not None else None,
                                       _ptr(sk, _f32p) if sk is not None else None,
                                       _ptr(gt, _f32p) if gt is not None else None,
                                       _ptr(out, _f64p), _ptr(lse, _f64p), _ptr(qrot, _f64p),
                                       kw.ctypes.data)
        if rc != 0:
            raise ValueError(f"oracle rejected the layer arguments (code {rc})")
        return {"out": out, "lse": lse, "qrot": qrot, "k_written": kw}

    def decode_tokens(self, *, layer_type: int, layout: int, window: int, rotary_dim: int,
                      rope_theta: float, context, q, k, v, kcache, vcache, sink=None, gate=None,
                      k_scale=None, v_scale=None):
        """T tokens per sequence in one step: q [B,T,Hq,D], k/v [B,T,Hkv,D] (uint16 bf16
        bits), caches as in decode_layer (updated in place), gate float32 [B,T,Hq] or
        None.  Returns dict(out [B,T,Hq,D] f64, lse [B,T,Hq] f64)."""
        for name, a in (("q", q), ("k", k), ("v", v)):
            if a.dtype != np.uint16 or not a.flags.c_contiguous or a.ndim != 4:
                raise ValueError(f"{name} must be C-contiguous uint16 [B, T, heads, D]")
        fp8 = kcache.dtype == np.uint8
        for name, a in (("kcache", kcache), ("vcache", vcache)):
            if a.dtype != (np.uint8 if fp8 else np.uint16) or not a.flags.c_contiguous:
                raise ValueError(f"{name} must be C-contiguous, uint16 bf16 bits or uint8 E4M3 codes")
        B, T, Hq, D = q.shape
        Hkv = k.shape[2]
        cap = kcache.shape[2]
        ctx = np.ascontiguousarray(context, dtype=np.int32)
        L = OrcLayer(B, Hq, Hkv, D, layer_type, layout, window, rotary_dim, float(rope_theta),
                     cap, Hkv * cap * D, KV_FP8_E4M3 if fp8 else KV_BF16)
        out = np.zeros((B, T, Hq, D))
        lse = np.zeros((B, T, Hq))
        sk = None if sink is None else np.ascontiguousarray(sink, dtype=np.float32)
        gt = None if gate is None else np.ascontiguousarray(gate, dtype=np.float32).reshape(B, T, Hq)
        ksc = None if k_scale is None else np.ascontiguousarray(k_scale, dtype=np.float32)
        vsc = None if v_scale is None else np.ascontiguousarray(v_scale, dtype=np.float32)
        if fp8 and (ksc is None or vsc is None):
            raise ValueError("an FP8 cache needs k_scale and v_scale")
        rc = self.lib.orc_decode_tokens(ctypes.byref(L), T, _ptr(ctx, _i32p), _ptr(q, _u16p), _ptr(k, _u16p),
                                        _ptr(v, _u16p), kcache.ctypes.data, vcache.ctypes.data,
                                        _ptr(ksc, _f32p) if ksc is not None else None,
                                        _ptr(vsc, _f32p) if vsc is not None else None,
                                        _ptr(sk, _f32p) if sk is not None else None,
                                        _ptr(gt, _f32p) if gt is not None else None,
                                        _ptr(out, _f64p), _ptr(lse, _f64p))
        if rc != 0:
            raise ValueError(f"oracle rejected the layer arguments (code {rc})")
        return {"out": out, "lse": lse}
