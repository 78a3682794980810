// Split-K flash-decoding for one layer of the hybrid model, and the LSE
// combine that folds in the per-head sink.
//
// The math is the scaled-dot-product attention of
// vllm_omni/edge/spark_export.py (`_Layer.forward`: scores = q.k/sqrt(d),
// softmax over keys, weights @ values, GQA by viewing q as (kv, group, d)),
// computed blockwise with an online softmax, which that page notes is
// numerically the same as one fused softmax (ring-branch comment).  The sink
// follows vllm/models/hy_v4/nvidia/flashmla_sparse.py
// (`HYV4FlashMLASparseImpl`): out *= exp(lse) / (exp(lse) + exp(sink)).
//
// Split pass: one CTA per (chunk of keys, kv head, sequence).  A producer warp
// streams the chunk's K and V rows through a 3-stage shared-memory ring with
// TMA tensor loads (128-byte swizzle, completion on an mbarrier); four
// consumer warps each take 8 keys of every 32-key stage, so each K/V row is
// read from HBM once for the whole GQA group.  Scores are kept in log2 units
// (q is pre-scaled by log2(e)/sqrt(d)).  The CTA writes an unnormalised
// partial (o, m, l) per query head.
//
// Combine: one CTA per (kv head, sequence) merges the partials of all chunks
// (and, for a sliding ring, the staged new entry), normalises, applies the
// sink, writes out/lse, and commits the staged ring entry to its slot now
// that every read of the ring has finished.
#include "hd_internal.h"

namespace hd {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kConsumerWarps = 4;
constexpr int kKeysPerWarp = kStageKeys / kConsumerWarps;  // 8
constexpr int kSplitThreads = (kConsumerWarps + 1) * 32;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // 1 s

// ------------------------------------------------------------ PTX helpers --
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Waits for the phase with the given parity; false once the time limit passed.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar, int x,
                                            int y, int z, int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void unpack_bf16x8(const uint4 &r, float (&f)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Number of cache keys the split pass scores for context c, or -1 (flagged)
// when c cannot be served.  Identical in the split and the combine kernels.
__device__ __forceinline__ int split_keys(int c, int key_set, int capacity, int window,
                                          int max_context, int chunk_keys, int max_chunks,
                                          int32_t *err, bool report) {
    int bit = 0, n = 0;
    if (c < 0) bit = HD_DEVERR_CONTEXT_NEGATIVE;
    else if (c > max_context) bit = HD_DEVERR_CONTEXT_PLAN;
    else if (key_set == KEYS_RING) n = min(c, capacity);
    else if (key_set == KEYS_ROLL) n = min(c + 1, window);
    else if (c >= capacity) bit = HD_DEVERR_CONTEXT_CAPACITY;
    else n = c + 1;
    if (!bit && (n + chunk_keys - 1) / chunk_keys > max_chunks) bit = HD_DEVERR_CONTEXT_PLAN;
    if (bit) {
        if (report) atomicOr(err, bit);
        return -1;
    }
    return n;
}

// --------------------------------------------------------------- split pass --
template <int G>
__global__ void __launch_bounds__(kSplitThreads, 2)
    attn_split_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const SplitArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint64_t *empty = full + kStages;

    const int chunk = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int n = split_keys(a.context[b], a.key_set, a.capacity, a.window, a.max_context,
                             a.chunk_keys, a.max_chunks, a.err,
                             chunk == 0 && kvh == 0 && threadIdx.x == 0);
    const int start = chunk * a.chunk_keys;
    if (n < 0 || start >= n) return;  // uniform over the CTA
    const int end = min(start + a.chunk_keys, n);
    const int nst = (end - start + kStageKeys - 1) / kStageKeys;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    float m[G], l[G], acc[G][8];
    if (warp == kConsumerWarps) {
        // Producer: one elected lane issues every load of the chunk.
        if (lane == 0) {
            for (int s = 0; s < nst; ++s) {
                const int slot = s % kStages;
                if (s >= kStages && !mbar_wait(&empty[slot], ((s / kStages) - 1) & 1)) {
                    atomicOr(a.err, HD_DEVERR_WAIT_TIMEOUT);
                    break;
                }
                uint8_t *st = smem + slot * kStageBytes;
                mbar_arrive_expect_tx(&full[slot], kStageBytes);
                const int row = start + s * kStageKeys;
#pragma unroll
                for (int j = 0; j < kBoxesPerRow; ++j)
                    tma_load_4d(st + j * kBoxBytes, &kmap, &full[slot], j * kBoxCols, row, kvh, b);
#pragma unroll
                for (int j = 0; j < kBoxesPerRow; ++j)
                    tma_load_4d(st + (kBoxesPerRow + j) * kBoxBytes, &vmap, &full[slot],
                                j * kBoxCols, row, kvh, b);
            }
        }
    } else {
        // Consumer: lane owns dims [8*lane, 8*lane+8), i.e. 16-byte chunk (lane&7)
        // of box (lane>>3); the 128-byte swizzle puts chunk j of row r at j^(r&7).
        const float qscale = kLog2e * 0.0625f;  // log2(e) / sqrt(256)
        float qv[G][8];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float4 *qp = reinterpret_cast<const float4 *>(
                a.q_rot + ((size_t)b * a.num_q_heads + kvh * G + h) * kHeadDim + lane * 8);
            const float4 x0 = qp[0], x1 = qp[1];
            qv[h][0] = x0.x * qscale; qv[h][1] = x0.y * qscale;
            qv[h][2] = x0.z * qscale; qv[h][3] = x0.w * qscale;
            qv[h][4] = x1.x * qscale; qv[h][5] = x1.y * qscale;
            qv[h][6] = x1.z * qscale; qv[h][7] = x1.w * qscale;
            m[h] = -INFINITY;
            l[h] = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[h][i] = 0.f;
        }
        const int box = lane >> 3, cidx = lane & 7;
        for (int s = 0; s < nst; ++s) {
            const int slot = s % kStages;
            if (!mbar_wait(&full[slot], (s / kStages) & 1)) {
                if (lane == 0) atomicOr(a.err, HD_DEVERR_WAIT_TIMEOUT);
                break;
            }
            const uint8_t *kst = smem + slot * kStageBytes + box * kBoxBytes;
            const uint8_t *vst = kst + kBoxesPerRow * kBoxBytes;
            // Keys are scored in sub-batches of KB so that the scores of a
            // sub-batch, q and the accumulators all stay in registers.
            constexpr int KB = G >= 8 ? 4 : kKeysPerWarp;
            const int key_base = start + s * kStageKeys + warp * kKeysPerWarp;
#pragma unroll
            for (int sb = 0; sb < kKeysPerWarp; sb += KB) {
                const int row0 = warp * kKeysPerWarp + sb;
                const int nvalid = min(KB, end - (key_base + sb));
                if (nvalid <= 0) break;  // warp-uniform
                float sc[KB][G];
#pragma unroll
                for (int r = 0; r < KB; ++r) {
                    const int row = row0 + r;
                    const uint4 raw =
                        *reinterpret_cast<const uint4 *>(kst + row * 128 + ((cidx ^ (row & 7)) << 4));
                    float kf[8];
                    unpack_bf16x8(raw, kf);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        float d = 0.f;
#pragma unroll
                        for (int i = 0; i < 8; ++i) d = fmaf(qv[h][i], kf[i], d);
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
                        sc[r][h] = (r < nvalid) ? d : -INFINITY;
                    }
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float mx = sc[0][h];
#pragma unroll
                    for (int r = 1; r < KB; ++r) mx = fmaxf(mx, sc[r][h]);
                    const float mn = fmaxf(m[h], mx);
                    const float alpha = fast_exp2(m[h] - mn);  // m = -inf -> 0
                    m[h] = mn;
                    l[h] *= alpha;
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[h][i] *= alpha;
#pragma unroll
                    for (int r = 0; r < KB; ++r) {
                        const float p = (r < nvalid) ? fast_exp2(sc[r][h] - mn) : 0.f;
                        sc[r][h] = p;
                        l[h] += p;
                    }
                }
#pragma unroll
                for (int r = 0; r < KB; ++r) {
                    if (r < nvalid) {  // rows past the key set may hold NaN: never touch them
                        const int row = row0 + r;
                        const uint4 raw = *reinterpret_cast<const uint4 *>(
                            vst + row * 128 + ((cidx ^ (row & 7)) << 4));
                        float vf[8];
                        unpack_bf16x8(raw, vf);
#pragma unroll
                        for (int h = 0; h < G; ++h)
#pragma unroll
                            for (int i = 0; i < 8; ++i) acc[h][i] = fmaf(sc[r][h], vf[i], acc[h][i]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
    }
    __syncthreads();  // every stage consumed: the ring is free for the warp merge

    float *red_o = reinterpret_cast<float *>(smem);             // [warps][G][256]
    float *red_m = red_o + kConsumerWarps * G * kHeadDim;       // [warps][G]
    float *red_l = red_m + kConsumerWarps * G;
    if (warp < kConsumerWarps) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float4 *dst = reinterpret_cast<float4 *>(red_o + (warp * G + h) * kHeadDim + lane * 8);
            dst[0] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
            dst[1] = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
            if (lane == 0) {
                red_m[warp * G + h] = m[h];
                red_l[warp * G + h] = l[h];
            }
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * kHeadDim; idx += blockDim.x) {
        const int h = idx / kHeadDim, d = idx % kHeadDim;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, red_m[w * G + h]);
        float o = 0.f, L = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float wt = fast_exp2(red_m[w * G + h] - M);
            o = fmaf(wt, red_o[(w * G + h) * kHeadDim + d], o);
            L = fmaf(wt, red_l[w * G + h], L);
        }
        const size_t pi = ((size_t)b * a.num_q_heads + kvh * G + h) * a.max_chunks + chunk;
        a.part_o[pi * kHeadDim + d] = o;
        if (d == 0) a.part_ml[pi] = make_float2(M, L);
    }
}

// ----------------------------------------------------------------- combine --
template <int G>
__global__ void __launch_bounds__(kHeadDim) attn_combine_kernel(const CombineArgs a) {
    const int kvh = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
    const int warp = d >> 5, lane = d & 31;
    __shared__ float red[kHeadDim / 32][G];
    __shared__ float s_new[G];
    const int c = a.context[b];
    const int n = split_keys(c, a.key_set, a.capacity, a.window, a.max_context, a.chunk_keys,
                             a.max_chunks, a.err, false);
    if (n < 0) {
        for (int h = 0; h < G; ++h) {
            const int hg = kvh * G + h;
            a.out[((size_t)b * a.num_q_heads + hg) * kHeadDim + d] = __float2bfloat16_rn(NAN);
            if (d == 0) a.lse[(size_t)b * a.num_q_heads + hg] = NAN;
        }
        return;
    }
    const int nchunks = (n + a.chunk_keys - 1) / a.chunk_keys;
    const bool ring = a.key_set == KEYS_RING;
    float vn = 0.f;
    if (ring) {
        const size_t e = ((size_t)b * a.num_kv_heads + kvh) * kHeadDim + d;
        const float kn = __bfloat162float(a.stage_k[e]);
        vn = __bfloat162float(a.stage_v[e]);
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float p = a.q_rot[((size_t)b * a.num_q_heads + kvh * G + h) * kHeadDim + d] * kn;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
            if (lane == 0) red[warp][h] = p;
        }
        __syncthreads();
        if (d < G) {
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < kHeadDim / 32; ++w) t += red[w][d];
            s_new[d] = t * (kLog2e * 0.0625f);
        }
        __syncthreads();
    }
#pragma unroll 1
    for (int h = 0; h < G; ++h) {
        const int hg = kvh * G + h;
        const size_t pb = ((size_t)b * a.num_q_heads + hg) * a.max_chunks;
        float M = ring ? s_new[h] : -INFINITY;
        for (int j = 0; j < nchunks; ++j) M = fmaxf(M, a.part_ml[pb + j].x);
        float o = 0.f, L = 0.f;
        for (int j = 0; j < nchunks; ++j) {
            const float2 ml = a.part_ml[pb + j];
            const float wt = exp2f(ml.x - M);
            L = fmaf(wt, ml.y, L);
            o = fmaf(wt, a.part_o[(pb + j) * kHeadDim + d], o);
        }
        if (ring) {
            const float wt = exp2f(s_new[h] - M);
            L += wt;
            o = fmaf(wt, vn, o);
        }
        const float lse = (M + log2f(L)) * kLn2;
        float f = 1.f;
        if (a.sink) f = 1.f / (1.f + expf(a.sink[hg] - lse));
        a.out[((size_t)b * a.num_q_heads + hg) * kHeadDim + d] = __float2bfloat16_rn(o / L * f);
        if (d == 0) a.lse[(size_t)b * a.num_q_heads + hg] = lse;
    }
    if (ring) {
        const int slot = c % a.capacity;
        const size_t e = ((size_t)b * a.num_kv_heads + kvh) * kHeadDim + d;
        const size_t o = (size_t)b * a.seq_stride + ((size_t)kvh * a.capacity + slot) * kHeadDim + d;
        a.cache_k[o] = a.stage_k[e];
        a.cache_v[o] = a.stage_v[e];
    }
}

template <int G>
cudaError_t split_g(const CUtensorMap *km, const CUtensorMap *vm, const SplitArgs &a, int batch,
                    cudaStream_t s) {
    static bool configured = false;
    const size_t smem = split_smem_bytes();
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(attn_split_kernel<G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    attn_split_kernel<G><<<dim3(a.max_chunks, a.num_kv_heads, batch), kSplitThreads, smem, s>>>(
        *km, *vm, a);
    return cudaGetLastError();
}

}  // namespace

size_t split_smem_bytes() { return 1024 + kStages * kStageBytes + 2 * kStages * sizeof(uint64_t); }

cudaError_t launch_split(const CUtensorMap *km, const CUtensorMap *vm, const SplitArgs &a, int batch,
                         int group, cudaStream_t s) {
    switch (group) {
    case 1: return split_g<1>(km, vm, a, batch, s);
    case 2: return split_g<2>(km, vm, a, batch, s);
    case 4: return split_g<4>(km, vm, a, batch, s);
    case 8: return split_g<8>(km, vm, a, batch, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_combine(const CombineArgs &a, int batch, int group, cudaStream_t s) {
    const dim3 grid(a.num_kv_heads, batch);
    switch (group) {
    case 1: attn_combine_kernel<1><<<grid, kHeadDim, 0, s>>>(a); break;
    case 2: attn_combine_kernel<2><<<grid, kHeadDim, 0, s>>>(a); break;
    case 4: attn_combine_kernel<4><<<grid, kHeadDim, 0, s>>>(a); break;
    case 8: attn_combine_kernel<8><<<grid, kHeadDim, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace hd
