// Partial Neox RoPE of q and the new k, and the store of the new K/V entry.
//
// vllm_omni/edge/spark_export.py, `_rope`: the leading rotary_dim dims are
// rotated as two halves (x1, x2) -> (x1*cos - x2*sin, x2*cos + x1*sin); the
// rest pass through.  `_angles` supplies cos/sin at the token's position,
// which is the number of previous tokens c.  The cache branches of
// `_Layer.forward` decide where the entry goes: append for full layers, the
// ring slot for this position (staged here, committed after the ring was
// read), or a window shifted by one (roll).
//
// q is rotated in fp32 (it only feeds the attention).  The stored key is the
// rotation from the fp32 table values, both products exact, rounded once to
// bf16 (rope_round.cuh: a binary32 evaluation when it is provably far from a
// rounding midpoint, else fp64 and round-to-odd).  An E4M3 cache stores
// e4m3(y / k_scale) of the fp64 rotation y (one fp64 division, one rounding)
// and e4m3(v / v_scale).
#include "e4m3.cuh"
#include "hd_internal.h"
#include "rope_round.cuh"

namespace hd {
namespace {

__device__ __forceinline__ void set_err(int32_t *err, int32_t bit) { atomicOr(err, bit); }

// Rotated value of dim d of one head vector x (bf16, global), fp32 path.
__device__ __forceinline__ float rope_f32(const __nv_bfloat16 *x, int d, int rot, const float2 *cs) {
    if (d >= rot) return __bfloat162float(x[d]);
    const int half = rot >> 1;
    const int i = d < half ? d : d - half;
    const float x1 = __bfloat162float(x[i]), x2 = __bfloat162float(x[i + half]);
    const float2 t = cs[i];
    return d < half ? fmaf(x1, t.x, -x2 * t.y) : fmaf(x2, t.x, x1 * t.y);
}

// Rotated value of dim d of the new key in fp64 (both products exact, one rounding).
__device__ __forceinline__ double rope_key_f64(const __nv_bfloat16 *x, int d, int rot, const float2 *cs) {
    if (d >= rot) return (double)__bfloat162float(x[d]);
    const int half = rot >> 1;
    const int i = d < half ? d : d - half;
    const double x1 = (double)__bfloat162float(x[i]), x2 = (double)__bfloat162float(x[i + half]);
    const double c = (double)cs[i].x, s = (double)cs[i].y;
    return d < half ? __dsub_rn(__dmul_rn(x1, c), __dmul_rn(x2, s)) : __dadd_rn(__dmul_rn(x2, c), __dmul_rn(x1, s));
}

// Stores dim d of the new entry at element offset o of the destination: the
// rotated key rounded once to bf16 and v bit for bit, or both as E4M3 codes.
__device__ __forceinline__ void store_entry(const RopeArgs &a, size_t o, int h, const __nv_bfloat16 *kh,
                                            const __nv_bfloat16 *vh, int d, const float2 *cs) {
    if (a.kv_type == KV_FP8) {
        const double y = rope_key_f64(kh, d, a.rotary_dim, cs);
        static_cast<uint8_t *>(a.dst_k)[o] = e4m3_quotient(y, (double)a.k_scale[h]);
        static_cast<uint8_t *>(a.dst_v)[o] = e4m3_quotient((double)__bfloat162float(vh[d]), (double)a.v_scale[h]);
    } else {
        __nv_bfloat16 k = kh[d];
        if (d < a.rotary_dim) {
            const int half = a.rotary_dim >> 1, i = d < half ? d : d - half;
            const float x1 = __bfloat162float(kh[i]), x2 = __bfloat162float(kh[i + half]);
            const float2 t = cs[i];
            k = __float2bfloat16_rn(d < half ? rotated_bf16(x1, t.x, x2, t.y) : rotated_bf16(x2, t.x, -x1, t.y));
        }
        static_cast<__nv_bfloat16 *>(a.dst_k)[o] = k;
        static_cast<__nv_bfloat16 *>(a.dst_v)[o] = vh[d];
    }
}

// Returns the context of sequence b, or -1 after flagging an unusable one.
__device__ __forceinline__ int checked_context(const RopeArgs &a, int b) {
    const int c = a.context[b];
    if (c < 0) {
        if (threadIdx.x == 0) set_err(a.err, HD_DEVERR_CONTEXT_NEGATIVE);
        return -1;
    }
    if (c > a.max_context) {
        if (threadIdx.x == 0) set_err(a.err, HD_DEVERR_CONTEXT_PLAN);
        return -1;
    }
    return c;
}

// One CTA per sequence: q of every head, and (full / ring) the new K/V entry.
__global__ void __launch_bounds__(256) rope_append_kernel(const RopeArgs a) {
    const int b = blockIdx.x;
    const int c = checked_context(a, b);
    if (c < 0) return;
    const int D = kHeadDim, rot = a.rotary_dim;
    const float2 *cs = a.table + (size_t)c * (rot >> 1);

    const __nv_bfloat16 *qb = a.q + (size_t)b * a.num_q_heads * D;
    float *qr = a.q_rot + (size_t)b * a.num_q_heads * D;
    for (int idx = threadIdx.x; idx < a.num_q_heads * D; idx += blockDim.x) {
        const int h = idx / D, d = idx % D;
        qr[idx] = rope_f32(qb + (size_t)h * D, d, rot, cs);
    }
    if (a.key_set == KEYS_ROLL) return;  // the roll kernel stores K/V
    int slot = 0;
    if (a.key_set == KEYS_FULL_CACHED) {
        if (c >= a.capacity) {
            if (threadIdx.x == 0) set_err(a.err, HD_DEVERR_CONTEXT_CAPACITY);
            return;
        }
        slot = c;
    }
    const __nv_bfloat16 *kb = a.k + (size_t)b * a.num_kv_heads * D;
    const __nv_bfloat16 *vb = a.v + (size_t)b * a.num_kv_heads * D;
    for (int idx = threadIdx.x; idx < a.num_kv_heads * D; idx += blockDim.x) {
        const int h = idx / D, d = idx % D;
        const size_t o = (size_t)b * a.seq_stride + ((size_t)h * a.capacity + slot) * D + d;
        store_entry(a, o, h, kb + (size_t)h * D, vb + (size_t)h * D, d, cs);
    }
}

// One CTA per (kv head, sequence) of a roll-layout sliding layer: shift the
// window down by one row once it is full, then write the new entry at the end.
// Rows move in groups of 256 / (16-byte chunks per row) -- 8 bf16 rows or 16
// E4M3 rows, one chunk per thread for K and for V: each group is read in full
// before any of it is overwritten, and the next group's first row is written
// only after the next read phase.
__global__ void __launch_bounds__(256) roll_window_kernel(const RopeArgs a) {
    const int h = blockIdx.x, b = blockIdx.y;
    const int c = checked_context(a, b);
    if (c < 0) return;
    const int D = kHeadDim, W = a.window;
    const int esize = kv_elem_bytes(a.kv_type);
    const size_t base = ((size_t)b * a.seq_stride + (size_t)h * a.capacity * D) * esize;   // bytes
    uint4 *K4 = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(a.dst_k) + base);
    uint4 *V4 = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(a.dst_v) + base);
    const int kChunksPerRow = kHeadDim * esize / 16;   // 32 or 16
    const int kRowsPerGroup = 256 / kChunksPerRow;      // 8 or 16 (blockDim.x == 256)
    int row_new = c;
    if (c >= W) {
        row_new = W - 1;
        const int r_local = threadIdx.x / kChunksPerRow, ch = threadIdx.x % kChunksPerRow;
        for (int r0 = 0; r0 < W - 1; r0 += kRowsPerGroup) {
            const int src = r0 + 1 + r_local;
            uint4 kk = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
            const bool live = src <= W - 1;
            if (live) {
                kk = K4[(size_t)src * kChunksPerRow + ch];
                vv = V4[(size_t)src * kChunksPerRow + ch];
            }
            __syncthreads();
            if (live) {
                K4[(size_t)(src - 1) * kChunksPerRow + ch] = kk;
                V4[(size_t)(src - 1) * kChunksPerRow + ch] = vv;
            }
            __syncthreads();
        }
    }
    const float2 *cs = a.table + (size_t)c * (a.rotary_dim >> 1);
    const __nv_bfloat16 *kh = a.k + ((size_t)b * a.num_kv_heads + h) * D;
    const __nv_bfloat16 *vh = a.v + ((size_t)b * a.num_kv_heads + h) * D;
    const size_t row_base = (size_t)b * a.seq_stride + ((size_t)h * a.capacity + row_new) * D;  // elements
    for (int d = threadIdx.x; d < D; d += blockDim.x) store_entry(a, row_base + d, h, kh, vh, d, cs);
}

}  // namespace

cudaError_t launch_rope_append(const RopeArgs &a, int batch, cudaStream_t s) {
    rope_append_kernel<<<batch, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_roll_window(const RopeArgs &a, int batch, cudaStream_t s) {
    roll_window_kernel<<<dim3(a.num_kv_heads, batch), 256, 0, s>>>(a);   // 256 threads: see the kernel
    return cudaGetLastError();
}

}  // namespace hd
