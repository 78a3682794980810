// One decode-attention layer of the hybrid model in one kernel: partial RoPE
// of q, split-K flash-decoding over the cached keys, and an LSE combine that
// scores the new entry, folds in the per-head sink and stores the entry.
//
// The math is the scaled-dot-product attention of
// vllm_omni/edge/spark_export.py (`_Layer.forward`: scores = q.k/sqrt(d),
// softmax over keys, weights @ values, GQA by viewing q as (kv, group, d)),
// computed blockwise with an online softmax, which that page notes is
// numerically the same as one fused softmax (ring-branch comment).  The new
// entry is scored apart from the cache, as that comment's two-key-set form
// does.  The sink follows vllm/models/hy_v4/nvidia/flashmla_sparse.py
// (`HYV4FlashMLASparseImpl`): out *= exp(lse) / (exp(lse) + exp(sink)).  The
// optional output gate of spark_export.py (`_Layer.forward`: each head's
// attention output times sigmoid of its gate logit) is applied in the same
// epilogue scale.
//
// Grid: one CTA per (chunk of cached keys, kv head, sequence).  The chunk's K
// and V rows stream through a shared-memory ring of 32 KiB stages (3 stages,
// or 6 with one CTA per SM) with TMA tensor loads (128-byte swizzle,
// completion on mbarriers); four consumer warps split every stage, so each K/V
// row is read from HBM once for the whole GQA group.  bf16 caches: 32-key
// stages, a dedicated producer warp.  E4M3 caches (per-kv-head scales):
// 64-key stages, the producer folded into the consumers (the last warp to
// release a slot refills it).  Scores are kept in log2 units (q is pre-scaled
// by log2(e)/sqrt(d)).  Consumers: CUDA-core FMA with warp-shuffle
// reductions, and tensor-core mma.sync with fp32 accumulation, where q is
// split into a high and a low part (bf16, or f16 for E4M3 caches) so the
// scores keep fp32 accuracy.  With MT, several tokens of a sequence are extra
// query rows (multi-token decode): 16 rows run on 64-key stages (16 keys per
// warp and call), and 32 rows -- more accumulators than registers hold -- on
// the 5th-generation tensor cores (tcgen05.mma, scores and outputs in tensor
// memory; see "Tensor-memory pass").
//
// A launch takes one layer (grid: chunks x kv heads x sequences) or, for a
// whole decode step, a table of up to kStepLayers layers in its parameters
// (a 1-D grid, each layer's CTAs a contiguous range): the layers of a step are
// independent, so one grid streams all their caches with no drain between layers.
// In a step grid a roll-layout layer reads its window before this step's
// shift and writes each row it read one row lower before releasing its stage
// (spark_export.py roll branch: drop the oldest entry, append the new one).
//
// Each CTA writes an unnormalised partial (o, m, l) per query row, then takes
// a ticket on a per-(sequence, kv head) counter.  The CTA that draws the last
// ticket -- every other chunk of that (sequence, kv head) has finished reading
// -- merges all partials and the new entries, writes out/lse, stores the new
// K/V entries (ring slot, append, or the rolled window's last row) and resets
// the counter.  Nothing waits on another CTA.
//
// This header holds the kernel and its launch templates; the translation units
// attn_decode.cu, attn_decode_fp8.cu, attn_step.cu and attn_step_fp8.cu each
// instantiate one family (cache type x single layer / step table).
#pragma once

#include <cuda_fp16.h>

#include "e4m3.cuh"
#include "hd_internal.h"
#include "rope_round.cuh"

// Build switches of the attention kernel (measured choices; see the comments at their use).
#ifndef HD_STEP_NEW_IN_EVERY_CTA
#define HD_STEP_NEW_IN_EVERY_CTA 1
#endif
#ifndef HD_STEP_ISSUE_EARLY
#define HD_STEP_ISSUE_EARLY 1
#endif
#ifndef HD_STEP_ARGS_IN_SMEM
#define HD_STEP_ARGS_IN_SMEM 0
#endif
#ifndef HD_STEP_FINISH
#define HD_STEP_FINISH 1
#endif

namespace hd {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kQScale = kLog2e * 0.0625f;   // log2(e) / sqrt(256)
constexpr int kConsumerWarps = 4;   // per CTA; 16-row multi-token passes run twice as many
// Who issues the copies.  bf16 single-layer kernels, multi-token passes and
// one-CTA-per-SM grids run a dedicated producer warp (lower latency for small
// grids: the batch-1 step 23.5 vs 27 us, the 16-row pass 3.12 vs 3.62 ms, and
// with 64-key stages 2.975 vs 3.002 ms although folding removed its spills).
// E4M3 kernels and the bf16 single-token step grids of two CTAs per SM fold the
// producer into the consumers (the last warp to release a slot refills it):
// four warps per CTA leave each thread up to 255 registers at two CTAs per SM,
// where five warps cap it at 168 -- the E4M3 consumer's conversions need them,
// and the bf16 step grid spilled at the cap (folded: 2.265 vs 2.303 ms at
// batch 64, 4.444 vs 4.498 ms at group 8).
__host__ __device__ constexpr bool own_producer(int kv, int nl, bool mt, bool deep) {
    return kv == KV_BF16 && (nl == 1 || mt || deep);
}
// With the tensor-memory consumer, a multi-token pass of 16 or 32 rows over a
// bf16 cache (one CTA per SM) runs on the tcgen05 tensor cores: four softmax
// warps per 16 rows, the producer warp and one warp that owns the tensor memory
// and issues the MMAs (see "Tensor-memory pass" below).
__host__ __device__ constexpr bool umma_pass(int g, int kv, bool mt, bool deep, int consumer) {
    return consumer == CONSUMER_UMMA && kv == KV_BF16 && mt && (g == 16 || g == 32) && deep;
}
// 16 query rows on mma.sync run one CTA per SM: eight consumer warps (two per row
// group of eight rows and stage half) keep as many warps per SM as two 8-row CTAs.
__host__ __device__ constexpr int consumer_warps(int g) { return g > kMaxGroup ? 2 * kConsumerWarps : kConsumerWarps; }
__host__ __device__ constexpr int layer_threads(int g, int kv, int nl, bool mt, bool deep,
                                                int consumer = CONSUMER_MMA) {
    return umma_pass(g, kv, mt, deep, consumer) ? (kConsumerWarps * (g / 16) + 2) * 32
                                      : (consumer_warps(g) + (own_producer(kv, nl, mt, deep) ? 1 : 0)) * 32;
}
// Shared memory of a tensor-memory pass of g rows past the common layout: two
// P^T buffers of 64 keys x g rows (bf16), the softmax warps' row maxima and sums,
// seventeen mbarriers and the tensor-memory address.
__host__ __device__ constexpr int umma_p_bytes(int g) { return 64 * g * 2; }
__host__ __device__ constexpr int umma_extra_bytes(int g) {
    return 128 + 2 * umma_p_bytes(g) + 3 * kConsumerWarps * g * 4 + 20 * 8 + 16;
}
// A ring of more than the default bytes: one CTA per SM; of at most two stages: three.
__host__ __device__ constexpr bool deep_ring(int s, int kv) { return s * kv_stage_bytes(kv) > kStages * kStageBytes; }
__host__ __device__ constexpr int ctas_per_sm(int s, int kv) {
    return deep_ring(s, kv) ? 1 : s * kv_stage_bytes(kv) <= kTripleStages * kStageBytes ? 3 : 2;
}
constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // 1 s
// Inside the stage ring (free once every stage is consumed): the warp buffers
// [warps][G][256] + (m, l) and the combine weights start at 0; this chunk's
// merged partial [G][256] + (m, l) sits past both.
constexpr int kOwnPartialOffset = 48 * 1024;
// Multi-token combine: the new entries of up to kMaxTokens tokens (K and V
// values, E4M3 codes) and the per-row weights of the new entries sit in the
// last kMtNewBytes of the (then free) stage ring.

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
// Non-blocking test of a phase (the tensor-memory pass's MMA warp polls two barriers).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
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
// Distributed shared memory of a thread-block cluster: the address of the same
// shared variable in CTA `rank` of the cluster, loads from it, and the
// cluster-wide barrier (release / acquire: shared-memory writes before it are
// visible to every CTA of the cluster after it).
__device__ __forceinline__ uint32_t dsmem_addr(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ float2 ld_dsmem_f2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float fast_log2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                              uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// D += A(16x8 bf16, row) * B(8x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(b0));
}
// m16n8k16 with f16 operands (the FP8 cache path: E4M3 converts to f16 exactly).
__device__ __forceinline__ void mma_16816_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
// Eight E4M3 codes (little-endian in two words) to floats.
__device__ __forceinline__ void unpack_e4m3x8(const uint2 &r, float (&f)[8]) {
    const uint32_t w[2] = {r.x, r.y};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t h = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i >> 1] >> (16 * (i & 1))));
        const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&h));
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
    }
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ void unpack_bf16x8(const uint4 &r, float (&f)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}
// ---------------------------------------------------------- tcgen05 helpers --
// Tensor memory: 128 lanes x 512 columns of 32-bit cells per SM.  An address is
// (lane << 16) | column; a warp reads the 32 lanes of its quarter (warp id % 4).
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {   // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {   // whole warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Shared-memory matrix descriptor: start, leading and stride byte offsets (16-byte
// units), the fixed version field, and the swizzle (2: 128-byte, 0: none).  For a
// 128-byte-swizzled K-major tile the stride offset steps 8-row groups and a k-step
// of 16 elements advances the start by 32 bytes inside the 1024-byte atom; for
// MN-major tiles the leading offset steps along M/N and the stride along K
// (128-byte swizzle), the other way round without swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swizzle << 61);
}
// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, K-major (0)
// or MN-major (1) operands, N / 8 and M / 16.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int m, int n, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
// D (+)= A B^T on the tensor cores, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)acc)
        : "memory");
}
// The mbarrier receives one arrival once every MMA this thread issued so far is complete.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
// 16 (32) consecutive columns of this thread's lane, then the wait for the load.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// Byte offset of element (operand row n, dim d) of the q operand: 2G rows (the
// high parts of rows 0..G-1, then their low parts) x 256 dims, K-major in column
// blocks of 64 dims x 2G rows x 128 bytes, 16-byte chunks swizzled.
template <int G>
__device__ __forceinline__ uint32_t umma_q_offset(int n, int d) {
    return (d >> 6) * (2 * G * 128) + n * 128 + ((((d >> 3) & 7) ^ (n & 7)) << 4) + 2 * (d & 7);
}
// Tensor-memory columns of a pass of g rows: scores S^T (2 buffers of 2g: high,
// low) at 0, O^T (2 buffers of 2g: two dim halves) at 4g; 8g in all.
__host__ __device__ constexpr uint32_t umma_cols(int g) { return 8u * (uint32_t)g; }

// q, once rotated and scaled, is kept as one 32-bit word per element: the value
// rounded to 16 bits in the low half and the remainder rounded to 16 bits in the
// high half -- bf16 with bf16 caches, f16 with E4M3 caches (the operand types of
// the tensor-core consumers) -- so hi + lo carries about 18 (bf16) or 22 (f16)
// significant bits.  The split is made once per element when q is rotated; the
// consumers build their operand fragments from it with byte permutes.
template <int KV>
__device__ __forceinline__ uint32_t q_split(float x) {
    if (KV == KV_FP8) {
        const __half h = __float2half_rn(x);
        const __half l = __float2half_rn(x - __half2float(h));
        return (uint32_t)__half_as_ushort(h) | ((uint32_t)__half_as_ushort(l) << 16);
    } else {
        const __nv_bfloat16 h = __float2bfloat16_rn(x);
        const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
        return (uint32_t)__bfloat16_as_ushort(h) | ((uint32_t)__bfloat16_as_ushort(l) << 16);
    }
}
template <int KV>
__device__ __forceinline__ float q_join(uint32_t w) {
    if (KV == KV_FP8)
        return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu))) +
               __half2float(__ushort_as_half((unsigned short)(w >> 16)));
    return __uint_as_float(w << 16) + __uint_as_float(w & 0xFFFF0000u);
}

// Byte offset of 16-byte chunk c (0..31 for bf16, 0..15 for E4M3) of row r in
// a stage's K or V region: box c/8, swizzled chunk (c%8)^(r%8) inside the
// 128-byte row.
template <int KV = KV_BF16>
__device__ __forceinline__ uint32_t tile_offset(int r, int c) {
    return (c >> 3) * kv_box_bytes(KV) + r * 128 + ((((c & 7) ^ (r & 7))) << 4);
}
// Transpose of an 8x8 matrix of 16-bit elements held one fragment per lane
// (lane l: row l/4, columns 2(l%4), 2(l%4)+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Scored cache keys of sequence context c, or -1 (and the error bit) when c
// cannot be served by this call.
__device__ __forceinline__ int cached_keys(const LayerArgs &a, int c, int *bit) {
    *bit = 0;
    if (c < 0) { *bit = HD_DEVERR_CONTEXT_NEGATIVE; return -1; }
    const int last = c + max(a.tokens, 1) - 1;   // position of the last new token
    if (last > a.max_context) { *bit = HD_DEVERR_CONTEXT_PLAN; return -1; }
    int n;
    switch (a.key_set) {
    case KEYS_RING: n = min(c, a.capacity); break;
    case KEYS_ROLL: n = min(c + 1, a.window); break;
    case KEYS_ROLL_SHIFT: n = min(c, a.window - 1); break;
    case KEYS_FULL_CACHED: n = c + 1; break;
    default: n = c; break;  // KEYS_FULL_PREV
    }
    if (n > a.capacity || (a.commit == COMMIT_APPEND && last >= a.capacity)) {
        *bit = HD_DEVERR_CONTEXT_CAPACITY;
        return -1;
    }
    if ((n + a.chunk_keys - 1) / a.chunk_keys > a.max_chunks) { *bit = HD_DEVERR_CONTEXT_PLAN; return -1; }
    if (a.key_set == KEYS_ROLL_SHIFT && (n > a.chunk_keys || a.window > a.capacity)) {   // one chunk shifts the window
        *bit = HD_DEVERR_CONTEXT_PLAN;
        return -1;
    }
    return n;
}

// ---------------------------------------------------------- the consumers --

// Ring window of the query rows of a multi-token step: row r (token t) must
// not see the t oldest ring entries -- positions c-511 .. c+t-512 left its
// window -- which sit in `cnt[r]` consecutive slots from slot `first`.
struct RowMask {
    int first = 0, cap = 1;
    const int *cnt = nullptr;   // [rows] in shared memory
    __device__ __forceinline__ bool hidden(int key, int count) const {
        int rel = key - first;
        if (rel < 0) rel += cap;
        return rel < count;
    }
};

// CUDA-core consumer: lane owns dims [8*lane, 8*lane+8) of every row; each
// score is a warp-shuffle reduction.  With an E4M3 cache the rows hold codes:
// scores take the K scale after the reduction and the output stays in V-code
// units (the combine applies the V scale).
template <int G, int KV>
struct FmaConsumer {
    static constexpr int kWK = kv_stage_keys(KV) / kConsumerWarps;   // keys per warp per stage
    float qv[G][8], m[G], l[G], acc[G][8];
    float kscale;

    __device__ void load_row(const uint8_t *st, int row, int lane, float (&f)[8]) const {
        if (KV == KV_FP8)
            unpack_e4m3x8(*reinterpret_cast<const uint2 *>(st + tile_offset<KV>(row, lane >> 1) + (lane & 1) * 8), f);
        else
            unpack_bf16x8(*reinterpret_cast<const uint4 *>(st + tile_offset<KV>(row, lane)), f);
    }

    __device__ void init(const uint32_t *qw, int lane, float k_scale) {
        kscale = k_scale;
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                qv[h][i] = q_join<KV>(qw[h * kHeadDim + lane * 8 + i]);
                acc[h][i] = 0.f;
            }
            m[h] = -INFINITY;
            l[h] = 0.f;
        }
    }

    __device__ void set_mask(const RowMask &, int) {}

    // Rows [row0, row0 + kWK) of a stage; the first nvalid are keys.
    __device__ void consume(const uint8_t *kst, const uint8_t *vst, int row0, int nvalid, int lane, int) {
        constexpr int KB = G >= 8 ? 4 : 8;  // keeps scores, q and acc in registers
#pragma unroll
        for (int sb = 0; sb < kWK; sb += KB) {
            const int nv = nvalid - sb;
            if (nv <= 0) break;  // warp-uniform
            float sc[KB][G];
#pragma unroll
            for (int r = 0; r < KB; ++r) {
                const int row = row0 + sb + r;
                float kf[8];
                load_row(kst, row, lane, kf);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float d = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) d = fmaf(qv[h][i], kf[i], d);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
                    if (KV == KV_FP8) d *= kscale;
                    sc[r][h] = (r < nv) ? d : -INFINITY;
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
                    const float p = (r < nv) ? fast_exp2(sc[r][h] - mn) : 0.f;
                    sc[r][h] = p;
                    l[h] += p;
                }
            }
#pragma unroll
            for (int r = 0; r < KB; ++r) {
                if (r < nv) {  // rows past the key set may hold NaN: never touch them
                    float vf[8];
                    load_row(vst, row0 + sb + r, lane, vf);
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[h][i] = fmaf(sc[r][h], vf[i], acc[h][i]);
                }
            }
        }
    }

    __device__ void store(float *red_o, float *red_m, float *red_l, int warp, int lane) const {
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
};

// Tensor-core consumer.  S = Q K^T with m16n8k16: rows 0..G-1 of the A tile
// hold bf16(q) and rows 8..8+G-1 hold bf16(q - bf16(q)), so row r plus row r+8
// of S is q.k to fp32 accuracy; the 8 keys of a warp are the N dimension and
// the K rows come straight from the swizzled TMA tile with ldmatrix.  The
// accumulator of S is, register for register, the B operand of
// O^T += V^T P^T (m16n8k8: dims on M, 8 keys on K, heads on N), whose A
// operand is V read with ldmatrix.trans.
//
// WIDE (16-row multi-token passes, 64-key stages of 8 KiB box columns): a call
// takes 16 keys as two 8-key tiles, so the score MMAs run as four independent
// chains, one softmax round covers 16 keys, and O^T += V^T P^T runs as m16n8k16
// (the two tiles' P fragments are its two B registers).
template <int G, bool MT = false, bool WIDE = false>
struct MmaConsumer {
    static constexpr int kWK = WIDE ? 16 : 8;   // keys per consume call
    static constexpr int kBoxB = (WIDE ? 2 : 1) * kv_box_bytes(KV_BF16);   // box column stride
    __device__ static __forceinline__ uint32_t off(int r, int c) {
        return (c >> 3) * kBoxB + r * 128 + ((((c & 7) ^ (r & 7))) << 4);
    }
    uint32_t qa[16][4];
    float o[16][4];   // O^T tile mt: rows dims 16mt + gid (+8), cols heads 2*t4 (+1)
    float m_run, l_run;  // for head gid; l_run sums this lane's keys only
    RowMask mask;
    int mcnt;            // MT: ring entries hidden from row gid

    __device__ void set_mask(const RowMask &m, int lane) {
        mask = m;
        mcnt = (lane >> 2) < G ? m.cnt[lane >> 2] : 0;
    }

    __device__ void init(const uint32_t *qw, int lane, float) {
        const int gid = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
            uint32_t r[4] = {0u, 0u, 0u, 0u};
            if (gid < G) {   // dims 16 ks + 2 t4 (+1) and the same + 8: high parts, then low parts
                const uint2 w0 = *reinterpret_cast<const uint2 *>(qw + gid * kHeadDim + 16 * ks + 2 * t4);
                const uint2 w8 = *reinterpret_cast<const uint2 *>(qw + gid * kHeadDim + 16 * ks + 2 * t4 + 8);
                r[0] = __byte_perm(w0.x, w0.y, 0x5410);
                r[1] = __byte_perm(w0.x, w0.y, 0x7632);
                r[2] = __byte_perm(w8.x, w8.y, 0x5410);
                r[3] = __byte_perm(w8.x, w8.y, 0x7632);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) qa[ks][j] = r[j];
        }
#pragma unroll
        for (int mt = 0; mt < 16; ++mt)
#pragma unroll
            for (int j = 0; j < 4; ++j) o[mt][j] = 0.f;
        m_run = -INFINITY;
        l_run = 0.f;
    }

    __device__ void consume(const uint8_t *kst, const uint8_t *vst, int row0, int nvalid, int lane, int key0) {
        if constexpr (WIDE) {
            consume16(kst, vst, row0, nvalid, lane, key0);
            return;
        }
        const int gid = lane >> 2, t4 = lane & 3;
        const int lrow = row0 + (lane & 7), lsub = lane >> 3;
        const uint32_t kbase = smem_u32(kst), vbase = smem_u32(vst);
        // Two accumulators (even / odd k-steps) halve the dependent MMA chain.
        float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kbase + off(lrow, 4 * p + lsub), b0, b1, b2, b3);
            mma_16816(s, qa[2 * p], b0, b1);
            mma_16816(s2, qa[2 * p + 1], b2, b3);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) s[j] += s2[j];
        bool ok0 = gid < G && 2 * t4 < nvalid, ok1 = gid < G && 2 * t4 + 1 < nvalid;
        if (MT) {
            ok0 = ok0 && !mask.hidden(key0 + 2 * t4, mcnt);
            ok1 = ok1 && !mask.hidden(key0 + 2 * t4 + 1, mcnt);
        }
        const float s0 = ok0 ? s[0] + s[2] : -INFINITY;
        const float s1 = ok1 ? s[1] + s[3] : -INFINITY;
        float mx = fmaxf(s0, s1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mn = fmaxf(m_run, mx);
        const float alpha = (mn == -INFINITY) ? 1.f : fast_exp2(m_run - mn);
        const float p0 = ok0 ? fast_exp2(s0 - mn) : 0.f;
        const float p1 = ok1 ? fast_exp2(s1 - mn) : 0.f;
        l_run = fmaf(l_run, alpha, p0 + p1);
        m_run = mn;
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
            const float a_lo = __shfl_sync(0xffffffffu, alpha, 8 * t4);      // head 2*t4
            const float a_hi = __shfl_sync(0xffffffffu, alpha, 8 * t4 + 4);  // head 2*t4+1
#pragma unroll
            for (int mt = 0; mt < 16; ++mt) {
                o[mt][0] *= a_lo;
                o[mt][1] *= a_hi;
                o[mt][2] *= a_lo;
                o[mt][3] *= a_hi;
            }
        }
        const uint32_t pb = pack_bf16(p0, p1);
        // Rows past the key set may hold NaN; 0 * NaN would poison the sum, so a
        // tile with fewer than kWK keys masks its V values (full tiles skip it).
        if (nvalid < kWK)
            pv(vbase, lrow, lsub, pb, (2 * t4 < nvalid ? 0x0000FFFFu : 0u) | (2 * t4 + 1 < nvalid ? 0xFFFF0000u : 0u));
        else
            pv(vbase, lrow, lsub, pb, 0xFFFFFFFFu);
    }

    __device__ __forceinline__ void pv(uint32_t vbase, int lrow, int lsub, uint32_t pb, uint32_t vmask) {
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(vbase + off(lrow, 4 * p + lsub), a0, a1, a2, a3);
            mma_1688(o[2 * p], a0 & vmask, a1 & vmask, pb);
            mma_1688(o[2 * p + 1], a2 & vmask, a3 & vmask, pb);
        }
    }

    // 16 keys row0..row0+15: tile A the first 8, tile B the next 8.
    __device__ void consume16(const uint8_t *kst, const uint8_t *vst, int row0, int nvalid, int lane, int key0) {
        const int gid = lane >> 2, t4 = lane & 3;
        const int lrow = row0 + (lane & 7), lsub = lane >> 3;
        const uint32_t kbase = smem_u32(kst), vbase = smem_u32(vst);
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sa2[4] = {0.f, 0.f, 0.f, 0.f};
        float sb[4] = {0.f, 0.f, 0.f, 0.f}, sb2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            ldsm_x4(kbase + off(lrow, 4 * p + lsub), a0, a1, a2, a3);
            ldsm_x4(kbase + off(lrow + 8, 4 * p + lsub), b0, b1, b2, b3);
            mma_16816(sa, qa[2 * p], a0, a1);
            mma_16816(sb, qa[2 * p], b0, b1);
            mma_16816(sa2, qa[2 * p + 1], a2, a3);
            mma_16816(sb2, qa[2 * p + 1], b2, b3);
        }
        // lane (gid, t4) scores keys 2t4, 2t4+1 (tile A) and 8+2t4, 9+2t4 (tile B) for row gid
        float x[4] = {sa[0] + sa2[0] + sa[2] + sa2[2], sa[1] + sa2[1] + sa[3] + sa2[3],
                      sb[0] + sb2[0] + sb[2] + sb2[2], sb[1] + sb2[1] + sb[3] + sb2[3]};
        const int kk[4] = {2 * t4, 2 * t4 + 1, 8 + 2 * t4, 9 + 2 * t4};
        bool ok[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            ok[i] = gid < G && kk[i] < nvalid;
            if (MT) ok[i] = ok[i] && !mask.hidden(key0 + kk[i], mcnt);
            x[i] = ok[i] ? x[i] : -INFINITY;
        }
        float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mn = fmaxf(m_run, mx);
        const float alpha = (mn == -INFINITY) ? 1.f : fast_exp2(m_run - mn);
        float pr[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) pr[i] = ok[i] ? fast_exp2(x[i] - mn) : 0.f;
        l_run = fmaf(l_run, alpha, (pr[0] + pr[1]) + (pr[2] + pr[3]));
        m_run = mn;
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
            const float a_lo = __shfl_sync(0xffffffffu, alpha, 8 * t4);      // head 2*t4
            const float a_hi = __shfl_sync(0xffffffffu, alpha, 8 * t4 + 4);  // head 2*t4+1
#pragma unroll
            for (int mt = 0; mt < 16; ++mt) {
                o[mt][0] *= a_lo;
                o[mt][1] *= a_hi;
                o[mt][2] *= a_lo;
                o[mt][3] *= a_hi;
            }
        }
        // P^T fragments of m16n8k16: keys 2t4, 2t4+1 (tile A) and 8+2t4, 9+2t4 (tile B) of head gid.
        const uint32_t pa = pack_bf16(pr[0], pr[1]), pb = pack_bf16(pr[2], pr[3]);
        // V^T tile mt (dims 16mt..16mt+15 x 16 keys) with ldmatrix.trans: lanes 0-7 the
        // first 8 keys at dims 16mt.., 8-15 the same keys at dims 16mt+8.., 16-31 the
        // next 8 keys likewise.  Rows past the key set may hold NaN (0 * NaN would
        // poison the sum), so a short call masks its V values.
        const int vrow = row0 + (lane & 7) + ((lane >> 4) << 3), vsub = (lane >> 3) & 1;
        uint32_t ma = 0xFFFFFFFFu, mb = 0xFFFFFFFFu;
        if (nvalid < kWK) {
            ma = (2 * t4 < nvalid ? 0x0000FFFFu : 0u) | (2 * t4 + 1 < nvalid ? 0xFFFF0000u : 0u);
            mb = (8 + 2 * t4 < nvalid ? 0x0000FFFFu : 0u) | (9 + 2 * t4 < nvalid ? 0xFFFF0000u : 0u);
        }
#pragma unroll
        for (int mt = 0; mt < 16; ++mt) {
            uint32_t v[4];
            ldsm_x4_trans(vbase + off(vrow, 2 * mt + vsub), v[0], v[1], v[2], v[3]);
            v[0] &= ma;
            v[1] &= ma;
            v[2] &= mb;
            v[3] &= mb;
            mma_16816(o[mt], v, pa, pb);
        }
    }

    __device__ void store(float *red_o, float *red_m, float *red_l, int warp, int lane) const {
        const int gid = lane >> 2, t4 = lane & 3;
        float l = l_run;
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        if (t4 == 0 && gid < G) {
            red_m[warp * G + gid] = m_run;
            red_l[warp * G + gid] = l;
        }
        const int h0 = 2 * t4, h1 = 2 * t4 + 1;
#pragma unroll
        for (int mt = 0; mt < 16; ++mt) {
            const int d = 16 * mt + gid;
            if (h0 < G) {
                red_o[(warp * G + h0) * kHeadDim + d] = o[mt][0];
                red_o[(warp * G + h0) * kHeadDim + d + 8] = o[mt][2];
            }
            if (h1 < G) {
                red_o[(warp * G + h1) * kHeadDim + d] = o[mt][1];
                red_o[(warp * G + h1) * kHeadDim + d + 8] = o[mt][3];
            }
        }
    }
};

// Tensor-core consumer for an E4M3 cache.  Codes convert exactly to f16
// (cvt.rn.f16x2.e4m3x2), so both products run as f16 MMAs (m16n8k16) with
// fp32 accumulation.  A warp takes 16 keys of a 64-key stage, and K is the A
// operand: S^T = K Q^T puts 16 keys on M and the q columns on N -- the f16
// high part of each head's q and, on the remaining columns, its low part
// (G <= 4: columns G..2G-1; G = 8: a second tile) -- so q costs two
// registers per k-step and one MMA covers 16 keys.
//
// K: lane (gid, t4) holds keys gid and gid + 8 and reads 16-byte chunks
// 2*t4 + (p & 1) + 8*(p >> 1) of both rows at step p (the eight lanes of a
// shared-memory phase then hit eight distinct chunks after the swizzle).
// Word j of a chunk is the A fragment of k-step 4p + j: dims (d, d+1) and
// (d+2, d+3) with d = 16*chunk + 4j; the q columns are built in init with the
// same dim order, which leaves every dot product unchanged.
//
// P: the S^T accumulator, packed to f16, is for each group of 8 keys one
// fragment of an 8x8 (keys x heads) matrix; movmatrix transposes it into the
// B operand of O^T += V^T P^T (m16n8k16: dims on M, 16 keys on K, heads on N).
// V: lane (gid, t4) reads chunk gid (and 8 + gid) of keys 2*t4, 2*t4+1,
// 2*t4+8, 2*t4+9; byte_perm pairs two keys' bytes of one dim, which is one
// E4M3x2 A register.  Tile mt covers, on row gid, dim
// 128*(mt / 8) + 16*gid + 2*(mt % 8) and, on row gid + 8, the next dim.
template <int G, bool MT = false>
struct Fp8MmaConsumer {
    static constexpr int NT = G == 8 ? 2 : 1;   // n-tiles of q columns
    static constexpr int kWK = 16;              // keys per warp per stage
    uint32_t qb[NT][16][2];
    float o[16][4];                              // O^T tile mt: dims (see above) x heads 2*t4 (+1)
    float m_run[2], l_run[2];                    // heads 2*t4 + e; l_run sums this lane's keys only
    float kscale;
    RowMask mask;
    int mcnt[2];                                 // MT: ring entries hidden from rows 2*t4 + e

    __device__ void set_mask(const RowMask &m, int lane) {
        mask = m;
#pragma unroll
        for (int e = 0; e < 2; ++e) mcnt[e] = 2 * (lane & 3) + e < G ? m.cnt[2 * (lane & 3) + e] : 0;
    }

    __device__ void init(const uint32_t *qw, int lane, float k_scale) {
        const int gid = lane >> 2, t4 = lane & 3;
        kscale = k_scale;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            // column gid of tile t: head and part (high or low f16 half of q)
            const bool lo = G == 8 ? t == 1 : gid >= G;
            const int head = G == 8 ? gid : (gid < G ? gid : gid - G);
            const bool used = G == 8 || gid < 2 * G;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const int chunk = 2 * t4 + (p & 1) + 8 * (p >> 1);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t r0 = 0u, r1 = 0u;
                    if (used) {   // four dims: their f16 high parts, or their low parts
                        const uint4 w = *reinterpret_cast<const uint4 *>(qw + head * kHeadDim + 16 * chunk + 4 * j);
                        const uint32_t sel = lo ? 0x7632u : 0x5410u;
                        r0 = __byte_perm(w.x, w.y, sel);
                        r1 = __byte_perm(w.z, w.w, sel);
                    }
                    qb[t][4 * p + j][0] = r0;
                    qb[t][4 * p + j][1] = r1;
                }
            }
        }
#pragma unroll
        for (int mt = 0; mt < 16; ++mt)
#pragma unroll
            for (int j = 0; j < 4; ++j) o[mt][j] = 0.f;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            m_run[e] = -INFINITY;
            l_run[e] = 0.f;
        }
    }

    __device__ void consume(const uint8_t *kst, const uint8_t *vst, int row0, int nvalid, int lane, int key0) {
        const int gid = lane >> 2, t4 = lane & 3;
        // S^T = K Q^T.  With one q tile, even and odd k-steps go to two accumulators
        // (half the dependent chain); two tiles are two chains already.
        float s[NT][4], s2[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int r = 0; r < 4; ++r) s[t][r] = s2[t][r] = 0.f;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int chunk = 2 * t4 + (p & 1) + 8 * (p >> 1);
            const uint4 ka = *reinterpret_cast<const uint4 *>(kst + tile_offset<KV_FP8>(row0 + gid, chunk));
            const uint4 kb = *reinterpret_cast<const uint4 *>(kst + tile_offset<KV_FP8>(row0 + gid + 8, chunk));
            const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w}, wb[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t a[4] = {e4m3x2_to_f16x2(static_cast<uint16_t>(wa[j] & 0xFFFFu)),
                                       e4m3x2_to_f16x2(static_cast<uint16_t>(wb[j] & 0xFFFFu)),
                                       e4m3x2_to_f16x2(static_cast<uint16_t>(wa[j] >> 16)),
                                       e4m3x2_to_f16x2(static_cast<uint16_t>(wb[j] >> 16))};
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if ((j & 1) && NT == 1)
                        mma_16816_f16(s2[t], a, qb[t][4 * p + j][0], qb[t][4 * p + j][1]);
                    else
                        mma_16816_f16(s[t], a, qb[t][4 * p + j][0], qb[t][4 * p + j][1]);
                }
            }
        }
        // Scores: registers 0/1 are key gid, 2/3 key gid + 8, for heads 2*t4 + e; add the low part.
        float sc[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) sc[r] = s[0][r] + s2[0][r];
        if (G == 8) {
#pragma unroll
            for (int r = 0; r < 4; ++r) sc[r] += s[NT - 1][r] + s2[NT - 1][r];
        } else if (G >= 2) {  // column c + G lives in lane t4 + G/2
#pragma unroll
            for (int r = 0; r < 4; ++r) sc[r] += __shfl_xor_sync(0xffffffffu, sc[r], G / 2);
        } else {              // G = 1: column 1 of the same lane
            sc[0] += sc[1];
            sc[2] += sc[3];
        }
        const bool k0 = gid < nvalid, k1 = gid + 8 < nvalid;
        float p[4], alpha[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const bool col = G == 8 || 2 * t4 + e < G;
            bool v0 = col && k0, v1 = col && k1;
            if (MT) {
                v0 = v0 && !mask.hidden(key0 + gid, mcnt[e]);
                v1 = v1 && !mask.hidden(key0 + gid + 8, mcnt[e]);
            }
            const float x0 = v0 ? sc[e] * kscale : -INFINITY;
            const float x1 = v1 ? sc[2 + e] * kscale : -INFINITY;
            float mx = fmaxf(x0, x1);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(m_run[e], mx);
            alpha[e] = (mn == -INFINITY) ? 1.f : fast_exp2(m_run[e] - mn);
            p[e] = v0 ? fast_exp2(x0 - mn) : 0.f;
            p[2 + e] = v1 ? fast_exp2(x1 - mn) : 0.f;
            l_run[e] = fmaf(l_run[e], alpha[e], p[e] + p[2 + e]);
            m_run[e] = mn;
        }
        if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
            for (int mt = 0; mt < 16; ++mt) {
                o[mt][0] *= alpha[0];
                o[mt][1] *= alpha[1];
                o[mt][2] *= alpha[0];
                o[mt][3] *= alpha[1];
            }
        }
        const uint32_t pb0 = movmatrix_trans(pack_f16(p[0], p[1]));   // keys 2*t4, +1 of head gid
        const uint32_t pb1 = movmatrix_trans(pack_f16(p[2], p[3]));   // keys 8 + 2*t4, +1
        // Rows past the key set may hold NaN codes; 0 * NaN would poison the sum,
        // so a tile with fewer than kWK keys masks its V values (full tiles skip it).
        if (nvalid < kWK) {
            const uint32_t m01 = (2 * t4 < nvalid ? 0x0000FFFFu : 0u) | (2 * t4 + 1 < nvalid ? 0xFFFF0000u : 0u);
            const uint32_t m89 = (2 * t4 + 8 < nvalid ? 0x0000FFFFu : 0u) | (2 * t4 + 9 < nvalid ? 0xFFFF0000u : 0u);
            pv(vst, row0, lane, pb0, pb1, m01, m89);
        } else {
            pv(vst, row0, lane, pb0, pb1, 0xFFFFFFFFu, 0xFFFFFFFFu);
        }
    }

    // O^T += V^T P^T over the tile's 16 keys; m01 / m89 mask the V values of keys
    // past the key set (all ones for a full tile, where the masks fold away).
    __device__ __forceinline__ void pv(const uint8_t *vst, int row0, int lane, uint32_t pb0, uint32_t pb1,
                                       uint32_t m01, uint32_t m89) {
        const int gid = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int chunk = 8 * half + gid;
            const uint4 v0 = *reinterpret_cast<const uint4 *>(vst + tile_offset<KV_FP8>(row0 + 2 * t4, chunk));
            const uint4 v1 = *reinterpret_cast<const uint4 *>(vst + tile_offset<KV_FP8>(row0 + 2 * t4 + 1, chunk));
            const uint4 v8 = *reinterpret_cast<const uint4 *>(vst + tile_offset<KV_FP8>(row0 + 2 * t4 + 8, chunk));
            const uint4 v9 = *reinterpret_cast<const uint4 *>(vst + tile_offset<KV_FP8>(row0 + 2 * t4 + 9, chunk));
            const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
            const uint32_t w8[4] = {v8.x, v8.y, v8.z, v8.w}, w9[4] = {v9.x, v9.y, v9.z, v9.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {   // dims 4w + 2q (row gid) and 4w + 2q + 1 (row gid + 8)
                    const uint32_t sel = q ? 0x7362u : 0x5140u;   // (key a, key b) byte pairs of two dims
                    const uint32_t x01 = __byte_perm(w0[w], w1[w], sel);
                    const uint32_t x89 = __byte_perm(w8[w], w9[w], sel);
                    const uint32_t a[4] = {e4m3x2_to_f16x2(static_cast<uint16_t>(x01 & 0xFFFFu)) & m01,
                                           e4m3x2_to_f16x2(static_cast<uint16_t>(x01 >> 16)) & m01,
                                           e4m3x2_to_f16x2(static_cast<uint16_t>(x89 & 0xFFFFu)) & m89,
                                           e4m3x2_to_f16x2(static_cast<uint16_t>(x89 >> 16)) & m89};
                    mma_16816_f16(o[8 * half + 2 * w + q], a, pb0, pb1);
                }
            }
        }
    }

    __device__ void store(float *red_o, float *red_m, float *red_l, int warp, int lane) const {
        const int gid = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float l = l_run[e];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            const int h = 2 * t4 + e;
            if (gid == 0 && h < G) {
                red_m[warp * G + h] = m_run[e];
                red_l[warp * G + h] = l;
            }
        }
        const int h0 = 2 * t4, h1 = 2 * t4 + 1;
#pragma unroll
        for (int mt = 0; mt < 16; ++mt) {
            const int d = 128 * (mt >> 3) + 16 * gid + 2 * (mt & 7);
            if (h0 < G)
                *reinterpret_cast<float2 *>(red_o + (warp * G + h0) * kHeadDim + d) = make_float2(o[mt][0], o[mt][2]);
            if (h1 < G)
                *reinterpret_cast<float2 *>(red_o + (warp * G + h1) * kHeadDim + d) = make_float2(o[mt][1], o[mt][3]);
        }
    }
};

// ------------------------------------------------------------- the kernel --

// G: query rows per kv head -- the GQA group, or with MT (multi-token) the
// group times a.tokens tokens of the same sequence, row r = token r / (G /
// a.tokens), head r % (G / a.tokens).  G = 16 (MT only) runs two row groups
// of 8 with eight consumer warps: warps 0-3 take rows 0-7 and warps 4-7 rows
// 8-15, each group splitting every stage's keys, so each warp keeps the 8-row
// consumer's registers.
// NL: layers in the parameter table (1: one layer, grid (chunks, kv heads,
// sequences); kStepLayers: a step, 1-D grid over the layers' CTA ranges).
template <int G, int CONSUMER, int SP, int KV, bool MT, int NL>
__global__ void __launch_bounds__(layer_threads(G, KV, NL, MT, deep_ring(SP, KV), CONSUMER), ctas_per_sm(SP, KV))
    attn_layer_kernel(const __grid_constant__ LaunchTable<NL> p) {
    // SP: the ring in 32 KiB stages.  A 16-row multi-token pass over a bf16 cache
    // takes them in pairs: 64-key stages, each K or V box column two 32-row boxes
    // one after the other (16 keys per consumer warp and stage, or the tcgen05 tile).
    constexpr bool kUmma = umma_pass(G, KV, MT, deep_ring(SP, KV), CONSUMER);
    constexpr bool kWide = kUmma || (HD_WIDE_MT && KV == KV_BF16 && MT && G == kMaxRowsMma && deep_ring(SP, KV));
    // A tensor-memory pass keeps K and V halves in rings of their own: (SP + 1) / 2
    // K slots and SP / 2 V slots (a K half is free once its scores are computed).
    constexpr int S = kUmma ? (SP + 1) / 2 : kWide ? SP / 2 : SP;        // ring slots (of K halves)
    constexpr int SV = kUmma ? SP / 2 : S;                               // slots of V halves
    constexpr int kRingBytes = SP * kv_stage_bytes(KV);                  // the whole ring
    constexpr int kStage = (kWide ? 2 : 1) * kv_stage_bytes(KV);        // bytes of one stage (K + V)
    constexpr int kKeys = (kWide ? 2 : 1) * kv_stage_keys(KV);          // keys per stage: 32 bf16, 64 E4M3 or wide
    constexpr int kBoxB = (kWide ? 2 : 1) * kv_box_bytes(KV);           // bytes of one box column of a stage
    constexpr int kBoxes = kv_boxes_per_row(KV);   // 128-byte boxes per K or V row
    // Rows of one TMA box (the host encodes the layer's tensor maps to match) and
    // boxes per box column of a stage.  A box of r rows fills r * 128 contiguous
    // bytes in the 128-byte swizzle, so two 32-row boxes and one 64-row box leave
    // the same layout.
    constexpr int kBoxRows = kWide ? kWideBoxRows : kv_stage_keys(KV);
    constexpr int kPieces = kKeys / kBoxRows;
    static_assert(kPieces * kBoxRows == kKeys, "whole boxes per stage");
    constexpr int kNThreads = layer_threads(G, KV, NL, MT, deep_ring(SP, KV), CONSUMER);
    constexpr bool kOwnProducer = own_producer(KV, NL, MT, deep_ring(SP, KV));
    constexpr int CW = kUmma ? kConsumerWarps * (G / 16) : consumer_warps(G);   // consumer (softmax) warps
    extern __shared__ uint8_t smem_raw[];
    // The ring starts on a 1024-byte boundary of the shared window (the 128-byte
    // swizzle repeats every 1024 bytes).  Offsetting the array pointer, rather than
    // rounding an integer address, keeps every pointer below in the shared space,
    // so the compiler emits shared-memory loads and stores for them.
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *q_s = reinterpret_cast<float *>(smem + kRingBytes);               // [G][256]
    float *knew_s = q_s + G * kHeadDim;                                        // [256]
    float *vnew_s = knew_s + kHeadDim;                                         // [256]
    float *kraw_s = vnew_s + kHeadDim;                                         // [256]
    float2 *tab_s = reinterpret_cast<float2 *>(kraw_s + kHeadDim);             // [128]
    float *misc = reinterpret_cast<float *>(tab_s + kHeadDim / 2);             // [32]
    uint64_t *full = reinterpret_cast<uint64_t *>(misc + 32);
    uint64_t *empty = full + S;
    int *flag_s = reinterpret_cast<int *>(empty + S);
    unsigned *rel_s = reinterpret_cast<unsigned *>(flag_s + 4);                // [S] slot releases (folded producer)
    uint8_t *code_s = reinterpret_cast<uint8_t *>(rel_s + 16);                 // [2][256] E4M3 new entry
    int *mcnt_s = reinterpret_cast<int *>(code_s + 2 * kHeadDim);               // [kMaxRows] MT ring masks
    // Tensor-memory pass: P^T buffers, the softmax warps' row maxima (two sets) and
    // sums, its mbarriers and the tensor-memory address (umma_extra_bytes).
    uint8_t *u_base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(mcnt_s + kMaxRows) + 127) & ~static_cast<uintptr_t>(127));
    constexpr int kPB = umma_p_bytes(G);                                            // one P^T buffer
    uint8_t *p_s = u_base;                                                           // [2][64 keys x G rows] bf16
    float *umax_s = reinterpret_cast<float *>(p_s + 2 * kPB);                       // [2][G / 16][4 warps][16]
    float *usum_s = umax_s + 2 * kConsumerWarps * G;                                // [softmax warps][16]
    // s[2] p[2] o[2] done x[2][2], then the V halves' full[3] and empty[3] (the K halves use full / empty)
    uint64_t *ubar = reinterpret_cast<uint64_t *>(usum_s + kConsumerWarps * G);
    uint64_t *fullv = ubar + 11, *emptyv = ubar + 14;
    uint32_t *taddr_s = reinterpret_cast<uint32_t *>(ubar + 20);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // This CTA's layer: the last one whose CTA range starts at or before it
    // (each lane tests one table entry; the ranges ascend).
    int layer = 0;
    if constexpr (NL > 1) {
        static_assert(NL <= 32, "one lane per table entry");
        const bool started = lane < p.num_layers && p.begin[lane] <= (int)blockIdx.x;
        layer = 31 - __clz(__ballot_sync(0xffffffffu, started));
    }
    const LayerLaunch &ll = p.layer[layer];
    // A step table is indexed at run time, so its layer's arguments are read
    // through a computed address (a single layer's from the parameters at fixed
    // offsets).  Copying them to shared memory once measured faster in the
    // register-capped bf16 kernels (two CTAs per SM) only while they had registers
    // to spare; it is off.
    constexpr bool kArgsInSmem = NL > 1 && HD_STEP_ARGS_IN_SMEM && KV == KV_BF16 && !kOwnProducer;
    __shared__ LayerArgs step_args_s;
    if constexpr (kArgsInSmem) {
        static_assert(sizeof(LayerArgs) % 4 == 0, "copied as words");
        for (int i = threadIdx.x; i < (int)(sizeof(LayerArgs) / 4); i += blockDim.x)
            reinterpret_cast<uint32_t *>(&step_args_s)[i] = reinterpret_cast<const uint32_t *>(&ll.a)[i];
        __syncthreads();
    }
    const LayerArgs &a = kArgsInSmem ? step_args_s : ll.a;
    int chunk, kvh, b;
    if constexpr (NL > 1) {
        const int local = (int)blockIdx.x - p.begin[layer];
        chunk = local % a.max_chunks;
        kvh = (local / a.max_chunks) % a.num_kv_heads;
        b = local / (a.max_chunks * a.num_kv_heads);
    } else {
        chunk = blockIdx.x;
        kvh = blockIdx.y;
        b = blockIdx.z;
    }
    // Programmatic dependent launch: the next grid in the stream may start as
    // soon as every CTA of this one has started.  Launched that way (only
    // behind another layer of the same step, see launch_layer), a CTA reads its
    // own layer's inputs and streams its own layer's cache -- nothing the
    // previous grid writes -- and waits for that grid (griddepcontrol.wait)
    // only before its first global write; in full stream order (wait_first) it
    // waits before anything else, which still hides the launch behind the
    // previous grid's last CTAs.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (a.wait_first) asm volatile("griddepcontrol.wait;" ::: "memory");
    // Tokens of this launch: one, or (MT) a.tokens tokens at positions c .. c + ntok - 1.
    const int ntok = MT ? a.tokens : 1;
    const int Gm = G / ntok;                               // model heads per kv head
    const int c = a.context[b] + (MT ? a.token0 : 0);
    // Row r of q / out / lse / gate in units of head vectors.
    auto qrow = [&](int r) -> size_t {
        if (!MT) return (size_t)b * a.num_q_heads + kvh * G + r;
        return ((size_t)b * a.total_tokens + a.token0 + r / Gm) * a.num_q_heads + kvh * Gm + r % Gm;
    };
    const float kscale = KV == KV_FP8 ? a.k_scale[kvh] : 1.f;
    const float vscale = KV == KV_FP8 ? a.v_scale[kvh] : 1.f;
    int bit = 0;
    const int n = cached_keys(a, c, &bit);
    if (n < 0) {
        if (chunk == 0) {  // this CTA reports and poisons the outputs of the group
            asm volatile("griddepcontrol.wait;" ::: "memory");
            if (threadIdx.x == 0) atomicOr(a.err, bit);
            for (int i = threadIdx.x; i < G * kHeadDim; i += blockDim.x) {
                const size_t r = qrow(i / kHeadDim);
                a.out[r * kHeadDim + i % kHeadDim] = __float2bfloat16_rn(NAN);
                if (i % kHeadDim == 0) a.lse[r] = NAN;
            }
        }
        return;
    }
    const int nchunks = max(1, (n + a.chunk_keys - 1) / a.chunk_keys);
    // Cluster launches: every CTA of the cluster takes part in its barriers, so a
    // chunk past the sequence's keys stays, with no keys, instead of leaving.
    const int clus = NL == 1 ? a.cluster : 0;
    if (chunk >= nchunks && clus <= 1) return;  // uniform over the CTA
    const int start = chunk * a.chunk_keys;
    const int end = min(start + a.chunk_keys, n);
    const int nst = end > start ? (end - start + kKeys - 1) / kKeys : 0;
    // A full rolled window read before its shift: key i is cache row i + 1.
    const int roff = (a.key_set == KEYS_ROLL_SHIFT && c >= a.window) ? 1 : 0;
    // After the pass the rolled window drops its sh oldest rows (rows sh.. move down
    // by sh) and takes the ntok new entries after them: once full, sh = ntok.
    const int sh = a.key_set == KEYS_ROLL_SHIFT ? max(0, min(c, a.window) + ntok - a.window) : 0;
    // New entries of the ntok tokens: values as scored (knew_t), V values (or
    // V codes' values for E4M3, vnew_t), codes, and per-row new-entry weights.
    uint8_t *mt_base = smem + kRingBytes - kMtNewBytes;
    float *knew_t = MT ? reinterpret_cast<float *>(mt_base) : knew_s;                      // [ntok][256]
    float *vnew_t = MT ? knew_t + kMaxTokens * kHeadDim : vnew_s;                            // [ntok][256]
    uint8_t *code_t = MT ? reinterpret_cast<uint8_t *>(vnew_t + kMaxTokens * kHeadDim) : code_s;
    const int vcode_off = MT ? kMaxTokens * kHeadDim : kHeadDim;                             // V codes
    constexpr int WN = MT ? kMaxTokens : 1;                                                  // wnew_t row stride
    // MT: per-row sink, gate, scale [3][kMaxRows] past the per-row new-entry weights
    float *rows_t = reinterpret_cast<float *>(code_t + 2 * kMaxTokens * kHeadDim) + kMaxRows * kMaxTokens;
    // Makes the new entries of the ntok tokens: the key rotated in fp64 and rounded
    // once to bf16, or quantised to E4M3 (fp64 rotation, one division, one
    // rounding; V too), each scored as stored; E4M3 V stays in code units.
    auto make_new_entries = [&]() {
        // One task per rotary pair (dims j and j + rotary_dim / 2 share their
        // inputs) and one per pass-through dim: one round over the CTA for a
        // fully rotated key.
        const int hr = a.rotary_dim >> 1;
        const int per = kHeadDim - hr;   // tasks per token
        for (int idx = threadIdx.x; idx < ntok * per; idx += blockDim.x) {
            const int t = idx / per, u = idx % per;
            const bool pair = u < hr;
            const int d0 = pair ? u : u + hr;
            // Raw k of token t at dim i and its rotary row (MT reads them here; a
            // single token's were fetched with the prologue's other inputs).
            const __nv_bfloat16 *kg = static_cast<const __nv_bfloat16 *>(a.new_k) +
                                      ((size_t)(b * a.total_tokens + a.token0 + t) * a.num_kv_heads + kvh) * kHeadDim;
            const __nv_bfloat16 *vg = static_cast<const __nv_bfloat16 *>(a.new_v) +
                                      ((size_t)(b * a.total_tokens + a.token0 + t) * a.num_kv_heads + kvh) * kHeadDim;
            auto kraw = [&](int i) -> float { return MT ? __bfloat162float(kg[i]) : kraw_s[i]; };
            auto vraw = [&](int i) -> float { return MT ? __bfloat162float(vg[i]) : vnew_s[i]; };
            // the key: rotated from the fp32 table -- in fp64 (exact products, one
            // rounding) for E4M3, rounded once to bf16 otherwise -- or passed
            // through / already staged
            double y0 = 0.0, y1 = 0.0;
            if (pair && a.new_kind == NEW_ROTATE) {
                const float x1 = kraw(u), x2 = kraw(u + hr);
                const float2 cs2 = MT ? a.table[(size_t)(c + t) * hr + u] : tab_s[u];
                if (KV == KV_FP8) {
                    const double cc = cs2.x, ss = cs2.y;
                    y0 = __dsub_rn(__dmul_rn((double)x1, cc), __dmul_rn((double)x2, ss));
                    y1 = __dadd_rn(__dmul_rn((double)x2, cc), __dmul_rn((double)x1, ss));
                } else {
                    y0 = rotated_bf16(x1, cs2.x, x2, cs2.y);
                    y1 = rotated_bf16(x2, cs2.x, -x1, cs2.y);
                }
            } else if (!(KV == KV_FP8 && a.new_kind == NEW_STAGED)) {
                y0 = kraw(d0);
                if (pair) y1 = kraw(u + hr);
            }
            for (int e = 0; e < (pair ? 2 : 1); ++e) {
                const int d = e ? u + hr : d0;
                const double y = e ? y1 : y0;
                const float vr = vraw(d);
                if (KV == KV_FP8) {
                    // E4M3 entry: quantise (one division, one rounding) unless staged;
                    // score it as stored (code * scale) and keep V in code units.
                    if (a.new_kind == NEW_ROTATE) {
                        code_t[t * kHeadDim + d] = e4m3_quotient(y, (double)kscale);
                        code_t[vcode_off + t * kHeadDim + d] = e4m3_quotient((double)vr, (double)vscale);
                    }
                    knew_t[t * kHeadDim + d] = e4m3_to_f32(code_t[t * kHeadDim + d]) * kscale;
                    vnew_t[t * kHeadDim + d] = e4m3_to_f32(code_t[vcode_off + t * kHeadDim + d]);
                } else {
                    // (a rotated key was rounded once to bf16; other values are bf16 already)
                    knew_t[t * kHeadDim + d] = (float)y;
                    vnew_t[t * kHeadDim + d] = vr;
                }
            }
        }
    };

    // Stage s of the chunk: one lane issues its K and V boxes into slot s % S.
    // A tensor-memory pass loads (and releases) a stage's K and V halves separately:
    // the K half is free once its scores are computed.
    auto issue_half = [&](int s, int v) {
        const int slot = v ? s % SV : s % S;
        uint8_t *st = smem + (v ? S + slot : slot) * (kStage / 2);
        uint64_t *bar = v ? &fullv[slot] : &full[slot];
        mbar_arrive_expect_tx(bar, kStage / 2);
        const int row = roff + start + s * kKeys;
#pragma unroll
        for (int j = 0; j < kBoxes; ++j)
#pragma unroll
            for (int h = 0; h < kPieces; ++h)
                tma_load_4d(st + j * kBoxB + h * kBoxRows * 128, v ? &ll.vmap : &ll.kmap, bar, j * kv_box_cols(KV),
                            row + h * kBoxRows, kvh, b);
    };
    auto issue_stage = [&](int s) {
        const int slot = s % S;
        uint8_t *st = smem + slot * kStage;
        mbar_arrive_expect_tx(&full[slot], kStage);
        const int row = roff + start + s * kKeys;
#pragma unroll
        for (int j = 0; j < kBoxes; ++j)
#pragma unroll
            for (int h = 0; h < kPieces; ++h)
                tma_load_4d(st + j * kBoxB + h * kBoxRows * 128, &ll.kmap, &full[slot], j * kv_box_cols(KV),
                            row + h * kBoxRows, kvh, b);
#pragma unroll
        for (int j = 0; j < kBoxes; ++j)
#pragma unroll
            for (int h = 0; h < kPieces; ++h)
                tma_load_4d(st + (kBoxes + j) * kBoxB + h * kBoxRows * 128, &ll.vmap, &full[slot],
                            j * kv_box_cols(KV), row + h * kBoxRows, kvh, b);
    };
    // Test hook: stages from a.drop_stage on are never issued (a copy that never arrives).
    auto droppable = [&](int s) { return a.drop_stage >= 0 && s >= a.drop_stage; };

    // Round 1 of the prologue: every thread requests its share of q (bf16 rows,
    // or fp32 rotated rows), the rotary row at position c and, for a
    // single-token pass, the new entry, the sinks and the gate logits, into
    // registers.  Then the thread that issues the copies initialises the
    // barriers and sends the first stages: the small requests reach memory ahead
    // of the stream, and the stream starts before they are back.
    const bool has_new = a.new_kind != NEW_NONE;
    // Where a single-token pass makes its new entry (rotation or quantisation,
    // score): in the prologue of every CTA, while the first stages are in flight
    // (whichever CTA combines then has it at hand, which shortens the critical
    // path: the bf16 batch-1 step grid 22.1 -> 21.75 us, the batch-64 one
    // unchanged since the key's rotation takes the binary32 path); in E4M3 step
    // grids (fp64 rotation and quantisation: +0.8 % at batch 64 in every CTA), and
    // with the switch off, only the CTA of a single-chunk sequence, the combining
    // CTA of a longer one making it after its ticket.
    constexpr bool kNewInEveryCta = NL == 1 || (HD_STEP_NEW_IN_EVERY_CTA && KV == KV_BF16);
    const bool new_early = !MT && has_new && (kNewInEveryCta || nchunks == 1 || clus > 1);
    const int half = a.rotary_dim >> 1;
    constexpr int kQLoads = (G * (kHeadDim / 4) + kNThreads - 1) / kNThreads;   // 16-byte q loads per thread
    const int nq16 = a.q_bf16 ? G * (kHeadDim / 8) : G * (kHeadDim / 4);
    uint4 qld[kQLoads];
#pragma unroll
    for (int k = 0; k < kQLoads; ++k) {
        const int i = threadIdx.x + k * kNThreads;
        if (i < nq16) {
            qld[k] = a.q_bf16 ? reinterpret_cast<const uint4 *>(a.q_bf16 + qrow(i / (kHeadDim / 8)) * kHeadDim)[i % (kHeadDim / 8)]
                              : reinterpret_cast<const uint4 *>(a.q_rot + qrow(i / (kHeadDim / 4)) * kHeadDim)[i % (kHeadDim / 4)];
        }
    }
    static_assert(kNThreads >= kHeadDim / 2, "one rotary pair per thread");
    const bool tab_ld = a.q_bf16 && !MT && (int)threadIdx.x < half;
    float2 tld = make_float2(0.f, 0.f);
    if (tab_ld) tld = a.table[(size_t)c * half + threadIdx.x];
    // the new entry: 16-byte loads, the K row then the V row (bf16: 32 each; E4M3 codes: 16 each)
    const bool codes_ld = KV == KV_FP8 && a.new_kind == NEW_STAGED;
    const int new_ld = new_early ? (codes_ld ? 32 : 64) : 0;
    uint4 nld = make_uint4(0u, 0u, 0u, 0u);
    if ((int)threadIdx.x < new_ld) {
        const int per = new_ld / 2, t = threadIdx.x;
        const size_t e = ((size_t)b * a.num_kv_heads + kvh) * kHeadDim * (codes_ld ? 1 : 2);
        const uint8_t *src = static_cast<const uint8_t *>(t < per ? a.new_k : a.new_v) + e;
        nld = reinterpret_cast<const uint4 *>(src)[t % per];
    }
    float sld = 0.f, gld = 0.f;
    if (!MT && (int)threadIdx.x < G) {
        if (a.sink) sld = a.sink[kvh * G + threadIdx.x];
        if (a.gate) gld = a.gate[(size_t)b * a.num_q_heads + kvh * G + threadIdx.x];
    }

    constexpr int kIssuer = kOwnProducer ? CW * 32 : 0;
    constexpr bool kIssueEarly = NL == 1 || HD_STEP_ISSUE_EARLY;
    const int early = min(S, nst);   // stages issued before the prologue ends
    auto issue_first = [&]() {
        if constexpr (kUmma) {   // as many K and V halves as their rings hold
            for (int s = 0; s < early && !droppable(s); ++s) issue_half(s, 0);
            for (int s = 0; s < min(SV, nst) && !droppable(s); ++s) issue_half(s, 1);
        } else {
            for (int s = 0; s < early && !droppable(s); ++s) issue_stage(s);
        }
    };
    if (threadIdx.x == kIssuer) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kUmma ? 1 : CW);   // tensor-memory pass: released by an MMA commit
            rel_s[s] = 0u;
        }
        if constexpr (kUmma) {
            static_assert(S <= 3, "three V-half barriers of each kind");
            for (int i = 0; i < 17; ++i)
                mbar_init(&ubar[i], i == 2 || i == 3 ? CW : (i >= 7 && i < 11) ? kConsumerWarps : 1);
        }
        fence_mbar_init();
        if (kIssueEarly) issue_first();
    }

    if constexpr (kUmma) {
        if (warp == CW + 1) {   // the MMA warp owns the tensor memory of the pass
            tmem_alloc(taddr_s, umma_cols(G));
            tc_fence_before();
        }
    }

    // Round 1 lands: q in shared memory as fp32, the rotary row, the new entry
    // (bf16 values as fp32, or E4M3 codes), the sinks and the gate logits.
#pragma unroll
    for (int k = 0; k < kQLoads; ++k) {
        const int i = threadIdx.x + k * kNThreads;
        if (i < nq16) {
            if (a.q_bf16) {
                float f[8];
                unpack_bf16x8(qld[k], f);
                float4 *dst = reinterpret_cast<float4 *>(q_s) + 2 * i;
                dst[0] = make_float4(f[0], f[1], f[2], f[3]);
                dst[1] = make_float4(f[4], f[5], f[6], f[7]);
            } else {
                reinterpret_cast<uint4 *>(q_s)[i] = qld[k];
            }
        }
    }
    if (tab_ld) tab_s[threadIdx.x] = tld;
    if ((int)threadIdx.x < new_ld) {
        const int per = new_ld / 2, t = threadIdx.x;
        if (codes_ld) {
            reinterpret_cast<uint4 *>(code_s + (t < per ? 0 : kHeadDim))[t % per] = nld;
        } else {
            float f[8];
            unpack_bf16x8(nld, f);
            float4 *dst = reinterpret_cast<float4 *>((t < per ? kraw_s : vnew_s) + (t % per) * 8);
            dst[0] = make_float4(f[0], f[1], f[2], f[3]);
            dst[1] = make_float4(f[4], f[5], f[6], f[7]);
        }
    }
    if (!MT && (int)threadIdx.x < G) {
        misc[2 * kMaxGroup + threadIdx.x] = sld;   // sink of row threadIdx.x
        misc[3 * kMaxGroup + threadIdx.x] = gld;   // gate logit of row threadIdx.x
    }
    __syncthreads();
    if (!kIssueEarly && threadIdx.x == kIssuer) issue_first();
    // Round 2: rotate each rotary pair in place (fp32; q only feeds the scores)
    // and scale every dim to log2 units.
    // (each element's word replaces its fp32 value in place)
    uint32_t *q_w = reinterpret_cast<uint32_t *>(q_s);
    if constexpr (kUmma) {
        // The B operand of S^T = K Q^T: operand rows 0..G-1 hold the bf16 high parts
        // of the q rows and rows G..2G-1 their low parts, K-major with the 128-byte
        // swizzle; a key's two scores are added after the MMA.  (One MMA costs the
        // same for N = 16 and N = 32, so the split costs no extra instructions.)
        // Every element is rotated and split into registers first, then written over
        // the fp32 rows.
        constexpr int kPer = (G * kHeadDim + kNThreads - 1) / kNThreads;
        uint32_t wv[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int e = threadIdx.x + k * kNThreads;
            float v = 0.f;
            if (e < G * kHeadDim) {
                const int r = e / kHeadDim, j = e % kHeadDim;
                v = q_s[e];
                if (a.q_bf16 && j < 2 * half) {
                    const int jj = j < half ? j : j - half;
                    const float2 t = a.table[(size_t)(c + r / Gm) * half + jj];   // position c + token
                    const float x1 = q_s[r * kHeadDim + jj], x2 = q_s[r * kHeadDim + jj + half];
                    v = j < half ? fmaf(x1, t.x, -x2 * t.y) : fmaf(x2, t.x, x1 * t.y);
                }
                v *= kQScale;
            }
            wv[k] = q_split<KV>(v);
        }
        __syncthreads();   // every read of the fp32 rows comes before the first write
        uint16_t *q16 = reinterpret_cast<uint16_t *>(q_s);
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int e = threadIdx.x + k * kNThreads;
            if (e < G * kHeadDim) {
                const int r = e / kHeadDim, j = e % kHeadDim;
                q16[umma_q_offset<G>(r, j) / 2] = (uint16_t)(wv[k] & 0xFFFFu);
                q16[umma_q_offset<G>(G + r, j) / 2] = (uint16_t)(wv[k] >> 16);
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // visible to the tensor cores
    } else if (a.q_bf16) {
        for (int p = threadIdx.x; p < G * half; p += blockDim.x) {
            const int r = p / half, j = p % half;
            const float2 t = MT ? a.table[(size_t)(c + r / Gm) * half + j] : tab_s[j];   // position c + token
            float *qr = q_s + r * kHeadDim;
            const float x1 = qr[j], x2 = qr[j + half];
            q_w[r * kHeadDim + j] = q_split<KV>(fmaf(x1, t.x, -x2 * t.y) * kQScale);
            q_w[r * kHeadDim + j + half] = q_split<KV>(fmaf(x2, t.x, x1 * t.y) * kQScale);
        }
        const int pass = kHeadDim - 2 * half;
        for (int i = threadIdx.x; i < G * pass; i += blockDim.x) {
            const int e = (i / pass) * kHeadDim + 2 * half + i % pass;
            q_w[e] = q_split<KV>(q_s[e] * kQScale);
        }
    } else {
        for (int i = threadIdx.x; i < G * kHeadDim; i += blockDim.x) q_w[i] = q_split<KV>(q_s[i] * kQScale);
    }
    // Single-token passes make the new entry here, in every CTA, while the first
    // stages are in flight (its inputs arrived with q): whichever CTA combines
    // the sequence then has it, and its score, at hand.
    if (new_early) make_new_entries();
    // MT sliding layers: row r (token t) does not see the oldest cached entries its
    // window has passed -- t of them once the window is full: ring slots from the
    // oldest one (slot c mod capacity), or the first keys of a rolled window read
    // before its shift (both windows hold window - 1 scored entries); rows of a
    // full layer see the whole cache.
    if (MT && threadIdx.x < G) {
        const int t = threadIdx.x / Gm;
        const int held = a.key_set == KEYS_RING ? a.capacity : a.window - 1;
        mcnt_s[threadIdx.x] =
            a.key_set == KEYS_RING || a.key_set == KEYS_ROLL_SHIFT ? (c >= held ? t : max(0, c + t - held)) : 0;
    }
    RowMask mask;
    mask.first = a.key_set == KEYS_RING && c >= a.capacity ? c % a.capacity : 0;
    mask.cap = a.capacity;
    mask.cnt = mcnt_s;
    __syncthreads();
    // The new entry's score per query row (log2 units: q is pre-scaled), kept
    // for the epilogue; the consumer warps take a row each.
    float *wnew_t = MT ? reinterpret_cast<float *>(code_t + 2 * kMaxTokens * kHeadDim) : misc + kMaxGroup;
    if (new_early && warp < CW) {
        for (int h = warp; h < G; h += CW) {
            float t = 0.f;
            for (int d = lane; d < kHeadDim; d += 32) t = fmaf(q_join<KV>(q_w[h * kHeadDim + d]), knew_t[d], t);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
            if (lane == 0) wnew_t[h] = t;
        }
    }

    // Row groups: RG groups of CG rows; each group's WPG warps split every stage.
    // (A tensor-memory pass leaves one partial of all G rows.)
    constexpr int RG = kUmma ? 1 : (G > 8 ? G / 8 : 1), CG = G / RG, WPG = kUmma ? 1 : CW / RG;
    constexpr int NRW = RG * WPG;                                // warp partials per row
    float *red_o = reinterpret_cast<float *>(smem);             // [NRW][CG][256], reuses the stage ring
    float *red_m = red_o + NRW * CG * kHeadDim;
    float *red_l = red_m + NRW * CG;
    if (kOwnProducer && warp == CW) {
        if (MT && sh > 0) {
            // Multi-token pass over a rolled window (bf16): the producer warp moves
            // each stage's rows down by sh once the stage has landed -- rows below
            // sh leave the window -- and only then refills the slot; every row
            // written was loaded by this or an earlier stage and later stages load
            // higher rows.  (This keeps the copy out of the consumers' registers.)
            constexpr int kChunks = kHeadDim * kv_elem_bytes(KV) / 16;   // 16-byte chunks per row
            const size_t seq = ((size_t)b * a.seq_stride + (size_t)kvh * a.capacity * kHeadDim) * kv_elem_bytes(KV);
            for (int s = 0; s < nst; ++s) {
                const int slot = s % S, vslot = s % SV;
                bool landed = mbar_wait(&full[slot], (s / S) & 1);
                if constexpr (kUmma) landed = landed && mbar_wait(&fullv[vslot], (s / SV) & 1);
                if (!__all_sync(0xffffffffu, landed)) {
                    if (lane == 0) atomicOr(a.err, HD_DEVERR_WAIT_TIMEOUT);
                    break;
                }
                const uint8_t *kst = kUmma ? smem + slot * (kStage / 2) : smem + slot * kStage;
                const uint8_t *vst = kUmma ? smem + (S + vslot) * (kStage / 2) : kst + kBoxes * kBoxB;
                const int key0 = start + s * kKeys, nrows = min(kKeys, end - key0);
                for (int i = lane; i < 2 * nrows * kChunks; i += 32) {
                    const int v = i >= nrows * kChunks, rem = i - v * nrows * kChunks;
                    const int r = rem / kChunks, ch = rem % kChunks, row = key0 + r + roff;
                    if (row < sh) continue;
                    const uint4 x = *reinterpret_cast<const uint4 *>(
                        (v ? vst : kst) + (ch >> 3) * kBoxB + r * 128 + ((((ch & 7) ^ (r & 7))) << 4));
                    *reinterpret_cast<uint4 *>(static_cast<uint8_t *>(v ? a.cache_v : a.cache_k) + seq +
                                               (size_t)(row - sh) * kHeadDim * kv_elem_bytes(KV) + 16 * ch) = x;
                }
                __syncwarp();
                int stop = 0;
                if constexpr (kUmma) {
                    // refill the K slot with stage s + S and the V slot with stage s + SV
                    if (lane == 0 && s + S < nst) {
                        if (droppable(s + S)) {
                            stop = 1;
                        } else if (!mbar_wait(&empty[slot], (s / S) & 1)) {
                            atomicOr(a.err, HD_DEVERR_WAIT_TIMEOUT);
                            stop = 1;
                        } else {
                            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                            issue_half(s + S, 0);
                        }
                    }
                    if (lane == 0 && !stop && s + SV < nst) {
                        if (droppable(s + SV)) {
                            stop = 1;
                        } else if (!mbar_wait(&emptyv[vslot], (s / SV) & 1)) {
                            atomicOr(a.err, HD_DEVERR_WAIT_TIMEOUT);
                            stop = 1;
                        } else {
                            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                            issue_half(s + SV, 1);
                        }
                    }
                } else if (lane == 0 && s + S < nst) {
                    if (droppable(s + S)) {
                        stop = 1;
                    } else if (!mbar_wait(&empty[slot], (s / S) & 1)) {
                        atomicOr(a.err, HD_DEVERR_WAIT_TIMEOUT);
                        stop = 1;
                    } else {
                        // this warp's reads of the slot come before the copy engine's write
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        issue_stage(s + S);
                    }
                }
                if (__shfl_sync(0xffffffffu, stop, 0)) break;
            }
        } else if (lane == 0) {
            if constexpr (kUmma) {
                // Tensor-memory pass: K and V halves have rings of their own; one lane
                // polls both (non-blocking) and refills each half as soon as its slot
                // is released, K first.
                int sk = min(S, nst), sv = min(SV, nst);   // next K and V halves to issue
                unsigned long long t_last = globaltimer_ns();
                unsigned spins = 0;
                while (sk < nst || sv < nst) {
                    bool did = false;
                    if (sk < nst) {
                        if (droppable(sk)) {
                            sk = nst;
                        } else if (mbar_test_wait(&empty[sk % S], ((sk / S) - 1) & 1)) {
                            issue_half(sk++, 0);
                            did = true;
                        }
                    }
                    if (sv < nst) {
                        if (droppable(sv)) {
                            sv = nst;
                        } else if (mbar_test_wait(&emptyv[sv % SV], ((sv / SV) - 1) & 1)) {
                            issue_half(sv++, 1);
                            did = true;
                        }
                    }
                    if (did) {
                        spins = 0;
                    } else if (++spins == 1) {
                        t_last = globaltimer_ns();
                    } else if ((spins & 63) == 0 && globaltimer_ns() - t_last > kWaitLimitNs) {
                        atomicOr(a.err, HD_DEVERR_WAIT_TIMEOUT);
                        break;
                    }
                }
            } else {
                // producer: one lane issues every load of the chunk
                for (int s = early; s < nst; ++s) {
                    if (droppable(s)) break;
                    const int slot = s % S;
                    if (s >= S && !mbar_wait(&empty[slot], ((s / S) - 1) & 1)) {
                        atomicOr(a.err, HD_DEVERR_WAIT_TIMEOUT);
                        break;
                    }
                    issue_stage(s);
                }
            }
        }
        __syncthreads();
        __syncthreads();
    } else if constexpr (kUmma) {
        // Tensor-memory pass (G = 16 or 32 query rows, 64-key stages).  Per stage s:
        //   S^T = K Q^T        tcgen05 M=64 (keys) x N=2G (rows: q high, q low) x K=256,
        //                      A = the K tile, B = the q operand; into columns 2G (s % 2)
        //   softmax            four warps per 16 rows: lane l < 16 of warp w scores key
        //                      16 (w % 4) + l for the group's rows (high + low); row maxima
        //                      over the group's warps through shared memory; P^T in bf16
        //                      to shared memory (MN-major, no swizzle)
        //   O^T_s = V^T P^T    M=128 (dims, two halves) x N=G x K=64 keys, A = the V tile
        //                      read MN-major; into columns 4G + 2G (s % 2), a fresh sum
        //   o = o * alpha_s + O^T_s   in the softmax warps' registers (lane = dim)
        // The MMA warp issues S^T of stage s + 1 before O^T of stage s, so the softmax of
        // one stage overlaps the MMAs of its neighbours; the commit after O^T_s releases
        // the slot.  Every wait is bounded and warp-uniform.
        if (warp == CW + 1) {
            tc_fence_after();
            const uint32_t tbase = *taddr_s;
            if (lane == 0) {
                constexpr uint32_t kIdQK = umma_idesc_bf16(64, 2 * G, 0, 0);
                constexpr uint32_t kIdPV = umma_idesc_bf16(128, G, 1, 1);
                // Descriptors are built once; an operand's k-step or slot only moves the
                // start-address field (16-byte units; shared addresses stay below 2^18),
                // so each MMA costs one 64-bit add per operand.
                const uint64_t kd0 = umma_desc(smem_u32(smem), 16, 1024, 2);                      // K halves
                const uint64_t vd0 = umma_desc(smem_u32(smem) + S * (kStage / 2), kBoxB, 1024, 2);  // V halves
                const uint64_t qd0 = umma_desc(smem_u32(q_s), 16, 1024, 2);
                // P^T: 8 keys x 8 rows per 128-byte core matrix, rows first (stride offset
                // 128), then keys (leading offset 16G bytes per 8 keys)
                const uint64_t pd0 = umma_desc(smem_u32(p_s), 16 * G, 128, 0);
                // Event loop: O^T of the oldest scored stage as soon as its P^T (and V
                // half) is there, else the scores of the next stage whose K half has
                // landed -- at most one stage ahead of the softmax warps (two score
                // buffers).  Each commit releases what its MMAs read.
                int q = 0, pv = 0;   // next stage to score, next stage to weight
                unsigned long long t_last = globaltimer_ns();
                unsigned spins = 0;
                while (pv < nst) {
                    if (pv < q && mbar_test_wait(&fullv[pv % SV], (pv / SV) & 1) &&
                        mbar_test_wait(&ubar[2 + (pv & 1)], (pv >> 1) & 1)) {
                        tc_fence_after();
                        const uint64_t vd = vd0 + (uint64_t)((pv % SV) * ((kStage / 2) >> 4));
                        const uint64_t pd = pd0 + (uint64_t)((pv & 1) * (kPB >> 4));
                        const uint32_t dO = tbase + 4 * G + (pv & 1) * 2 * G;
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int t = 0; t < 4; ++t)
                                umma_bf16(dO + h * G, vd + (uint64_t)((2 * h * kBoxB + t * 2048) >> 4),
                                          pd + (uint64_t)((t * 32 * G) >> 4), kIdPV, t > 0);
                        umma_commit(&ubar[4 + (pv & 1)]);
                        umma_commit(&emptyv[pv % SV]);
                        ++pv;
                        spins = 0;
                    } else if (q < nst && q <= pv + 1 && mbar_test_wait(&full[q % S], (q / S) & 1)) {
                        tc_fence_after();
                        const uint64_t kd = kd0 + (uint64_t)((q % S) * ((kStage / 2) >> 4));
                        const uint32_t dS = tbase + (q & 1) * 2 * G;
#pragma unroll
                        for (int kk = 0; kk < 16; ++kk)
                            umma_bf16(dS, kd + (uint64_t)(((kk >> 2) * kBoxB + (kk & 3) * 32) >> 4),
                                      qd0 + (uint64_t)(((kk >> 2) * (2 * G * 128) + (kk & 3) * 32) >> 4), kIdQK, kk > 0);
                        umma_commit(&ubar[q & 1]);
                        umma_commit(&empty[q % S]);
                        ++q;
                        spins = 0;
                    } else if (++spins == 1) {
                        t_last = globaltimer_ns();
                    } else if ((spins & 63) == 0 && globaltimer_ns() - t_last > kWaitLimitNs) {
                        atomicOr(a.err, HD_DEVERR_WAIT_TIMEOUT);
                        break;
                    }
                }
                // every MMA issued above is complete before the tensor memory is freed
                umma_commit(&ubar[6]);
                if (!mbar_wait(&ubar[6], 0)) atomicOr(a.err, HD_DEVERR_WAIT_TIMEOUT);
            }
            __syncwarp();
            __syncthreads();
            __syncthreads();
        } else {
            // Warp w: rows r0..r0+15 of its group, keys 16 (w % 4) .. + 15 of each stage
            // (tensor-memory lanes of its quarter).
            constexpr int R = 16;
            const int grp = warp / kConsumerWarps, quarter = warp % kConsumerWarps, r0 = R * grp;
            tc_fence_after();
            const uint32_t tl = *taddr_s + ((uint32_t)(32 * quarter) << 16);   // this warp's lane quarter
            const int kl = lane & 15;
            // Lane l (and l + 16) keeps row l's running maximum and the last stage's
            // weight; the rows' values reach every lane by shuffles (registers are
            // scarce with 32 rows: ten warps leave 168 per thread).
            float m_row = -INFINITY, al_row = 1.f;
            float l_part[R], o_acc[2 * R];
            int cnt[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                l_part[r] = 0.f;
                o_acc[r] = 0.f;
                o_acc[R + r] = 0.f;
                cnt[r] = mcnt_s[r0 + r];
            }
            bool ok = true;
            auto fail = [&]() {
                if (lane == 0) atomicOr(a.err, HD_DEVERR_WAIT_TIMEOUT);
                ok = false;
            };
            // O^T of stage ps joins the running sum (its rows rescaled by alpha_ps, row
            // r's weight held by lane r).
            float al_prev = 1.f;
            auto fold = [&](int ps) -> bool {
                if (!__all_sync(0xffffffffu, mbar_wait(&ubar[4 + (ps & 1)], (ps >> 1) & 1))) return false;
                tc_fence_after();
                float ov[2 * R];
                const uint32_t oc = tl + 4 * G + (ps & 1) * 2 * G + r0;   // half h at + h * G
                if constexpr (G == 16) {
                    tmem_ld32(oc, ov);
                } else {
                    tmem_ld16(oc, ov);
                    tmem_ld16(oc + G, ov + R);
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float al = __shfl_sync(0xffffffffu, al_prev, r);
                    o_acc[r] = fmaf(o_acc[r], al, ov[r]);
                    o_acc[R + r] = fmaf(o_acc[R + r], al, ov[R + r]);
                }
                return true;
            };
            for (int s = 0; s < nst; ++s) {
                const int sb = s & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(&ubar[sb], (s >> 1) & 1))) {
                    fail();
                    break;
                }
                tc_fence_after();
                float x[R];
                {
                    float hl[2 * R];
                    const uint32_t sc = tl + sb * 2 * G + r0;   // high parts; the low ones at + G
                    if constexpr (G == 16) {
                        tmem_ld32(sc, hl);
                    } else {
                        tmem_ld16(sc, hl);
                        tmem_ld16(sc + G, hl + R);
                    }
#pragma unroll
                    for (int r = 0; r < R; ++r) x[r] = hl[r] + hl[R + r];
                }
                const int kin = 16 * quarter + kl;   // this lane's key in the stage (lanes < 16)
                const int key = start + s * kKeys + kin;
                const bool live = lane < 16 && key < end;
#pragma unroll
                for (int r = 0; r < R; ++r) x[r] = live && !(MT && mask.hidden(key, cnt[r])) ? x[r] : -INFINITY;
                // Row maxima over the warp's 16 keys: each step halves the rows a lane
                // keeps (lane bit 8, 4, 2, 1), so lane l ends with row l.
                float mx[R];
#pragma unroll
                for (int r = 0; r < R; ++r) mx[r] = x[r];
#pragma unroll
                for (int w = R / 2; w >= 1; w >>= 1) {
                    const bool up = (lane & w) != 0;
#pragma unroll
                    for (int i = 0; i < w; ++i) {
                        const float keep = up ? mx[i + w] : mx[i], send = up ? mx[i] : mx[i + w];
                        mx[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, w));
                    }
                }
                float *um = umax_s + (sb * (G / 16) + grp) * kConsumerWarps * R;
                uint64_t *xbar = &ubar[7 + 2 * sb + grp];
                if (lane < 16) um[quarter * R + lane] = mx[0];
                __syncwarp();
                if (lane == 0) mbar_arrive(xbar);
                if (!__all_sync(0xffffffffu, mbar_wait(xbar, (s >> 1) & 1))) {
                    fail();
                    break;
                }
                float mst = um[kl];
#pragma unroll
                for (int w = 1; w < kConsumerWarps; ++w) mst = fmaxf(mst, um[w * R + kl]);
                // row kl: new maximum and the weight of what came before
                const float mn_row = fmaxf(m_row, mst);
                al_row = mn_row == -INFINITY ? 1.f : fast_exp2(m_row - mn_row);
                m_row = mn_row;
                float pv[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float mn = __shfl_sync(0xffffffffu, mn_row, r);
                    const float alpha = __shfl_sync(0xffffffffu, al_row, r);
                    pv[r] = x[r] == -INFINITY ? 0.f : fast_exp2(x[r] - mn);
                    l_part[r] = fmaf(l_part[r], alpha, pv[r]);
                }
                // P^T of this stage, MN-major without swizzle: key k, row j at
                // (k / 8) * 16G + (k % 8) * 16 + (j / 8) * 128 + (j % 8) * 2.
                if (lane < 16) {
                    uint8_t *pb = p_s + sb * kPB + (kin >> 3) * 16 * G + (kin & 7) * 16 + (r0 >> 3) * 128;
                    *reinterpret_cast<uint4 *>(pb) = make_uint4(pack_bf16(pv[0], pv[1]), pack_bf16(pv[2], pv[3]),
                                                                pack_bf16(pv[4], pv[5]), pack_bf16(pv[6], pv[7]));
                    *reinterpret_cast<uint4 *>(pb + 128) = make_uint4(pack_bf16(pv[8], pv[9]), pack_bf16(pv[10], pv[11]),
                                                                      pack_bf16(pv[12], pv[13]), pack_bf16(pv[14], pv[15]));
                }
                // Rows past the key set may hold NaN; 0 * NaN would poison O^T, so the V
                // rows of a short stage are cleared (the K rows only reach masked scores).
                const int nv = end - (start + s * kKeys);
                if (nv < kKeys) {
                    if (!__all_sync(0xffffffffu, mbar_wait(&fullv[s % SV], (s / SV) & 1))) {   // the V half has landed
                        fail();
                        break;
                    }
                    uint8_t *vst = smem + (S + s % SV) * (kStage / 2);
                    const int per = (kKeys - nv) * 8;   // 16-byte chunks per box column
                    for (int i = threadIdx.x; i < kBoxes * per; i += CW * 32)
                        *reinterpret_cast<uint4 *>(vst + (i / per) * kBoxB + (nv + (i % per) / 8) * 128 + (i % 8) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // P^T and V for the tensor cores
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ubar[2 + sb]);
                if (s >= 1 && !fold(s - 1)) {
                    fail();
                    break;
                }
                al_prev = al_row;
            }
            if (ok && nst > 0 && !fold(nst - 1)) fail();
            tc_fence_before();
            // This chunk's row sums over the 64 lanes that scored: lane l < 16 ends with row l.
#pragma unroll
            for (int w = R / 2; w >= 1; w >>= 1) {
                const bool up = (lane & w) != 0;
#pragma unroll
                for (int i = 0; i < w; ++i) {
                    const float keep = up ? l_part[i + w] : l_part[i], send = up ? l_part[i] : l_part[i + w];
                    l_part[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
                }
            }
            if (lane < 16) usum_s[warp * R + lane] = l_part[0];
            __syncthreads();   // every stage consumed: the ring is free for the partial
            const int d0 = 32 * quarter + lane;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                red_o[(r0 + r) * kHeadDim + d0] = o_acc[r];
                red_o[(r0 + r) * kHeadDim + 128 + d0] = o_acc[R + r];
            }
            if (quarter == 0 && lane < R) {
                float l = 0.f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) l += usum_s[(grp * kConsumerWarps + w) * R + lane];
                red_m[r0 + lane] = m_row;
                red_l[r0 + lane] = l;
            }
            __syncthreads();
        }
    } else {
        using Mma = typename std::conditional<KV == KV_FP8, Fp8MmaConsumer<CG, MT>, MmaConsumer<CG, MT, kWide>>::type;
        typename std::conditional<CONSUMER == CONSUMER_MMA, Mma, FmaConsumer<CG, KV>>::type cons;
        constexpr int kCallKeys = decltype(cons)::kWK;          // keys per consume call
        constexpr int kSpan = kKeys / WPG;                        // keys of a stage per warp
        const int rg = warp / WPG, kpart = warp % WPG;
        cons.init(q_w + rg * CG * kHeadDim, lane, kscale);
        if (MT) {
            RowMask gm = mask;
            gm.cnt = mcnt_s + rg * CG;
            cons.set_mask(gm, lane);
        }
        for (int s = 0; s < nst; ++s) {
            const int slot = s % S;
            if (!mbar_wait(&full[slot], (s / S) & 1)) {
                if (lane == 0) atomicOr(a.err, HD_DEVERR_WAIT_TIMEOUT);
                break;
            }
            const uint8_t *kst = smem + slot * kStage;
#pragma unroll
            for (int sub = 0; sub < kSpan; sub += kCallKeys) {
                const int row0 = kpart * kSpan + sub;
                const int nvalid = min(kCallKeys, end - (start + s * kKeys + row0));
                if (nvalid > 0)
                    cons.consume(kst, kst + kBoxes * kBoxB, row0, nvalid, lane, start + s * kKeys + row0);
            }
            // Rolled window: this warp's rows of the stage (cache rows key + roff) move
            // down by sh rows before the slot is released; rows below sh leave the
            // window.  Every row written was loaded by this or an earlier stage; later
            // stages load higher rows.  A single token moves a full window by one row
            // (sh = roff); several tokens by the entries that leave it -- with bf16
            // caches the producer warp does that, with E4M3 caches the first row group
            // (the groups read the same keys).  A layer kernel launched as a
            // programmatic dependent follows another layer of the step, which never
            // touches this cache, so these writes need no dependency wait.
            if constexpr (!MT) {
                if (roff) {
                    const int key0 = start + s * kKeys + kpart * kSpan;
                    const int nrows = min(kSpan, end - key0);
                    constexpr int kChunks = kHeadDim * kv_elem_bytes(KV) / 16;   // 16-byte chunks per row
                    const size_t seq = ((size_t)b * a.seq_stride + (size_t)kvh * a.capacity * kHeadDim) *
                                       kv_elem_bytes(KV);
                    for (int i = lane; i < 2 * nrows * kChunks; i += 32) {
                        const int v = i >= nrows * kChunks, rem = i - v * nrows * kChunks;
                        const int r = rem / kChunks, ch = rem % kChunks;
                        const uint4 x = *reinterpret_cast<const uint4 *>(
                            kst + v * kBoxes * kv_box_bytes(KV) + tile_offset<KV>(kpart * kSpan + r, ch));
                        uint8_t *dst = static_cast<uint8_t *>(v ? a.cache_v : a.cache_k) + seq +
                                       (size_t)(key0 + r) * kHeadDim * kv_elem_bytes(KV) + 16 * ch;
                        *reinterpret_cast<uint4 *>(dst) = x;
                    }
                }
            } else if constexpr (!kOwnProducer) {   // no producer warp to do it
                if (sh > 0 && rg == 0) {
                    const int key0 = start + s * kKeys + kpart * kSpan;
                    const int nrows = min(kSpan, end - key0);
                    constexpr int kChunks = kHeadDim * kv_elem_bytes(KV) / 16;
                    const size_t seq = ((size_t)b * a.seq_stride + (size_t)kvh * a.capacity * kHeadDim) *
                                       kv_elem_bytes(KV);
                    for (int i = lane; i < 2 * nrows * kChunks; i += 32) {
                        const int v = i >= nrows * kChunks, rem = i - v * nrows * kChunks;
                        const int r = rem / kChunks, ch = rem % kChunks;
                        const int row = key0 + r + roff;
                        if (row < sh) continue;
                        const int rr = kpart * kSpan + r;
                        const uint4 x = *reinterpret_cast<const uint4 *>(
                            kst + v * kBoxes * kBoxB + (ch >> 3) * kBoxB + rr * 128 + ((((ch & 7) ^ (rr & 7))) << 4));
                        uint8_t *dst = static_cast<uint8_t *>(v ? a.cache_v : a.cache_k) + seq +
                                       (size_t)(row - sh) * kHeadDim * kv_elem_bytes(KV) + 16 * ch;
                        *reinterpret_cast<uint4 *>(dst) = x;
                    }
                }
            }
            __syncwarp();  // orders every lane's reads of the slot before lane 0's release
            if (lane == 0) {
                if (kOwnProducer) {
                    mbar_arrive(&empty[slot]);
                } else {
                    // Folded producer: the last of the consumer warps to release the slot
                    // refills it with stage s + S (release / acquire through the counter,
                    // then a proxy fence before the async-proxy write).
                    __threadfence_block();
                    const unsigned prev = atomicAdd(&rel_s[slot], 1u);
                    if (prev % CW == CW - 1 && s + S < nst && !droppable(s + S)) {
                        __threadfence_block();
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        issue_stage(s + S);
                    }
                }
            }
        }
        __syncthreads();  // every stage consumed: the ring is free for the warp merge
        cons.store(red_o, red_m, red_l, warp, lane);
        __syncthreads();
    }
    if constexpr (kUmma) {
        if (warp == CW + 1) {   // every tensor-memory read and MMA is complete (barriers above)
            tc_fence_after();
            tmem_dealloc(*taddr_s, umma_cols(G));
        }
    }

    // Per query row: this chunk's maximum M and sum L over the warps of the
    // row's group, and each warp's weight 2^(m_w - M) (shared memory only).
    // Partials: G rows per (sequence, kv head), num_kv_heads * G rows per sequence.
    const size_t pbase = ((size_t)b * a.num_kv_heads * G + kvh * G) * a.max_chunks;
    // this chunk's partial, the warp weights and the rows' lse sit past the warp buffers
    constexpr int kRedBytes = (NRW * CG * kHeadDim + 2 * NRW * CG) * (int)sizeof(float);
    // (a two-stage ring, single-token only, has its own partial right past the warp buffers)
    constexpr int kRedEnd = (kRedBytes + 1023) / 1024 * 1024;
    constexpr int kOwnOff = kRingBytes <= kTripleStages * kStageBytes ? kRedEnd
                            : kRedBytes <= kOwnPartialOffset          ? kOwnPartialOffset
                                                                      : kRedEnd;
    static_assert(kOwnOff + G * (kHeadDim + 2 + WPG + 1 + kMaxCluster) * (int)sizeof(float) <=
                      kRingBytes - (MT ? kMtNewBytes : 0),
                  "warp buffers, own partial and the multi-token entries fit the ring");
    static_assert(!MT || kRingBytes > kTripleStages * kStageBytes, "multi-token passes keep at least three stages");
    float *own_o = reinterpret_cast<float *>(smem + kOwnOff);   // [G][256]
    float2 *own_ml = reinterpret_cast<float2 *>(own_o + G * kHeadDim);    // [G]
    float *wwarp = reinterpret_cast<float *>(own_ml + G);                 // [G][WPG]
    float *lse_s = wwarp + G * WPG;                                        // [G]
    float *wclu = lse_s + G;                                               // [G][kMaxCluster] cluster weights
    float *sink_s = MT ? rows_t : misc + 2 * kMaxGroup;                  // [G]
    float *gate_s = MT ? rows_t + kMaxRows : misc + 3 * kMaxGroup;       // [G]
    float *head_s = MT ? rows_t + 2 * kMaxRows : misc;   // [G] scale = sink factor * gate / L
    // A single-token CTA holding the only chunk of its sequence finishes the rows
    // itself: the new entry joins the maximum and the sum here.  (In step grids
    // this measured 0.1-0.7 % faster than the general combine once their
    // two-CTA kernels folded the producer and had registers to spare.)
    const bool finish = (NL == 1 || HD_STEP_FINISH) && !MT && nchunks == 1 && clus <= 1;
    if (threadIdx.x < G) {
        const int h = threadIdx.x, w0 = (h / CG) * WPG, hr = h % CG;
        float M = -INFINITY;
#pragma unroll
        for (int w = w0; w < w0 + WPG; ++w) M = fmaxf(M, red_m[w * CG + hr]);
        const float s_new = finish && has_new ? wnew_t[h] : -INFINITY;
        M = fmaxf(M, s_new);
        float L = 0.f;
#pragma unroll
        for (int w = w0; w < w0 + WPG; ++w) {
            const float m = red_m[w * CG + hr];
            const float wt = (m == -INFINITY) ? 0.f : fast_exp2(m - M);
            wwarp[h * WPG + (w - w0)] = wt;
            L = fmaf(wt, red_l[w * CG + hr], L);
        }
        if (finish) {
            const float w_new = has_new ? fast_exp2(s_new - M) : 0.f;
            wnew_t[h] = w_new;
            L += w_new;
            const float lse = (M + fast_log2(L)) * kLn2;
            // exp(lse) / (exp(lse) + exp(sink)) = 1 / (1 + 2^((sink - lse) * log2 e))
            float f = a.sink ? 1.f / (1.f + fast_exp2((sink_s[h] - lse) * kLog2e)) : 1.f;
            // output gate: sigmoid(g) = 1 / (1 + 2^(-g * log2 e)); lse is not gated
            if (a.gate) f *= 1.f / (1.f + fast_exp2(-gate_s[h] * kLog2e));
            head_s[h] = f / L * vscale;   // FP8: partials and the new value are in V-code units
            lse_s[h] = lse;
        } else {
            own_ml[h] = make_float2(M, L);
        }
    }
    __syncthreads();

    // Stores the new entries now that every chunk of this (sequence, kv head) has read the cache.
    auto store_new_entries = [&]() {
        if (!has_new || a.commit == COMMIT_NONE) return;
        for (int idx = threadIdx.x; idx < ntok * kHeadDim; idx += blockDim.x) {
            const int t = idx / kHeadDim, d = idx % kHeadDim;
            const int slot = a.commit == COMMIT_RING   ? (c + t) % a.capacity
                             : a.commit == COMMIT_ROLL ? min(c, a.window) + t - sh
                                                       : c + t;
            const size_t o = (size_t)b * a.seq_stride + ((size_t)kvh * a.capacity + slot) * kHeadDim + d;
            if (KV == KV_FP8) {
                static_cast<uint8_t *>(a.cache_k)[o] = code_t[t * kHeadDim + d];
                static_cast<uint8_t *>(a.cache_v)[o] = code_t[vcode_off + t * kHeadDim + d];
            } else {  // exact: the values are bf16 values
                static_cast<__nv_bfloat16 *>(a.cache_k)[o] = __float2bfloat16_rn(knew_t[t * kHeadDim + d]);
                static_cast<__nv_bfloat16 *>(a.cache_v)[o] = __float2bfloat16_rn(vnew_t[t * kHeadDim + d]);
            }
        }
    };
    // Row h of the warps' outputs at dims [4 dq, 4 dq + 4), weighted by the warp weights.
    const float4 *red_o4 = reinterpret_cast<const float4 *>(red_o);
    auto warp_sum = [&](int h, int dq) -> float4 {
        const int w0 = (h / CG) * WPG, hr = h % CG;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < WPG; ++w) {
            const float wt = wwarp[h * WPG + w];
            const float4 v = red_o4[((w0 + w) * CG + hr) * (kHeadDim / 4) + dq];
            o.x = fmaf(wt, v.x, o.x);
            o.y = fmaf(wt, v.y, o.y);
            o.z = fmaf(wt, v.z, o.z);
            o.w = fmaf(wt, v.w, o.w);
        }
        return o;
    };
    auto store_out = [&](int h, int dq, const float (&o)[4]) {
        const float sc = head_s[h];
        __nv_bfloat16 r[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) r[i] = __float2bfloat16_rn(o[i] * sc);
        uint2 packed;
        packed.x = (uint32_t)__bfloat16_as_ushort(r[0]) | ((uint32_t)__bfloat16_as_ushort(r[1]) << 16);
        packed.y = (uint32_t)__bfloat16_as_ushort(r[2]) | ((uint32_t)__bfloat16_as_ushort(r[3]) << 16);
        *reinterpret_cast<uint2 *>(a.out + qrow(h) * kHeadDim + 4 * dq) = packed;
    };

    // (single-layer deep-ring launches only: the host sends clusters nowhere else)
    if constexpr (NL == 1 && !MT && kRingBytes > kStages * kStageBytes) {
        if (clus > 1) {
            // Cluster combine: CTA r of the cluster holds chunk r's partial in its
            // shared memory.  After the cluster barrier every CTA reads all chunks'
            // (m, l) pairs, forms the rows' maximum, weights, sum and lse (the new
            // entry included), and merges its own slice of the dims from every
            // chunk's partial -- all before the dependency wait, since none of it
            // touches global memory; then it stores its slice of out, and rank 0
            // stores lse and the new entry.  A last barrier keeps every CTA's
            // shared memory alive until the others have read it.
            for (int i = threadIdx.x; i < G * (kHeadDim / 4); i += blockDim.x)
                reinterpret_cast<float4 *>(own_o)[i] = warp_sum(i / (kHeadDim / 4), i % (kHeadDim / 4));
            cluster_sync_all();
            const int rank = chunk;   // the cluster spans the chunk dimension
            if (threadIdx.x < G) {
                const int h = threadIdx.x;
                float2 ml_r[kMaxCluster];
                float M = has_new ? wnew_t[h] : -INFINITY;
#pragma unroll
                for (int r = 0; r < kMaxCluster; ++r) {
                    ml_r[r] = make_float2(-INFINITY, 0.f);
                    if (r < clus) ml_r[r] = ld_dsmem_f2(dsmem_addr(own_ml + h, r));
                    M = fmaxf(M, ml_r[r].x);
                }
                float L = 0.f;
#pragma unroll
                for (int r = 0; r < kMaxCluster; ++r) {
                    const float w = (ml_r[r].x == -INFINITY) ? 0.f : fast_exp2(ml_r[r].x - M);
                    if (r < clus) wclu[h * kMaxCluster + r] = w;
                    L = fmaf(w, ml_r[r].y, L);
                }
                const float w_new = has_new ? fast_exp2(wnew_t[h] - M) : 0.f;
                L += w_new;
                wnew_t[h] = w_new;
                const float lse = (M + fast_log2(L)) * kLn2;
                float f = a.sink ? 1.f / (1.f + fast_exp2((sink_s[h] - lse) * kLog2e)) : 1.f;
                if (a.gate) f *= 1.f / (1.f + fast_exp2(-gate_s[h] * kLog2e));
                head_s[h] = f / L * vscale;
                lse_s[h] = lse;
            }
            __syncthreads();
            // this CTA's float4 columns of every row
            const int col0 = rank * (kHeadDim / 4) / clus, col1 = (rank + 1) * (kHeadDim / 4) / clus;
            const int ncol = col1 - col0;
            constexpr int kTasks = (G * (kHeadDim / 8) + kNThreads - 1) / kNThreads;   // clusters have >= 2 CTAs
            float res[kTasks][4];
#pragma unroll
            for (int k = 0; k < kTasks; ++k) {
                const int i = threadIdx.x + k * kNThreads;
                if (i < G * ncol) {
                    const int h = i / ncol, dq = col0 + i % ncol;
                    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int r = 0; r < clus; ++r) {
                        const float w = wclu[h * kMaxCluster + r];
                        const float4 v = ld_dsmem_f4(dsmem_addr(reinterpret_cast<const float4 *>(own_o) + h * 64 + dq, r));
                        o.x = fmaf(w, v.x, o.x);
                        o.y = fmaf(w, v.y, o.y);
                        o.z = fmaf(w, v.z, o.z);
                        o.w = fmaf(w, v.w, o.w);
                    }
                    if (has_new) {
                        const float wn = wnew_t[h];
                        const float4 vn = reinterpret_cast<const float4 *>(vnew_t)[dq];
                        o.x = fmaf(wn, vn.x, o.x);
                        o.y = fmaf(wn, vn.y, o.y);
                        o.z = fmaf(wn, vn.z, o.z);
                        o.w = fmaf(wn, vn.w, o.w);
                    }
                    res[k][0] = o.x;
                    res[k][1] = o.y;
                    res[k][2] = o.z;
                    res[k][3] = o.w;
                }
            }
            asm volatile("griddepcontrol.wait;" ::: "memory");
#pragma unroll
            for (int k = 0; k < kTasks; ++k) {
                const int i = threadIdx.x + k * kNThreads;
                if (i < G * ncol) store_out(i / ncol, col0 + i % ncol, res[k]);
            }
            if (rank == 0) {
                if (threadIdx.x < G) a.lse[qrow(threadIdx.x)] = lse_s[threadIdx.x];
                store_new_entries();
            }
            cluster_sync_all();
            return;
        }
    }

    // Everything above only read this layer's own inputs and cache.  The first
    // global write (partials, tickets, outputs, the stored entry) waits for the
    // previous grid in the stream to complete and its writes to be visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (finish) {
        // out = (sum of the warps' weighted rows + w_new * v_new) * scale, lse, the new entry.
        for (int i = threadIdx.x; i < G * (kHeadDim / 4); i += blockDim.x) {
            const int h = i / (kHeadDim / 4), dq = i % (kHeadDim / 4);
            const float4 o4 = warp_sum(h, dq);
            float o[4] = {o4.x, o4.y, o4.z, o4.w};
            if (has_new) {
                const float wn = wnew_t[h];
                const float4 vn = reinterpret_cast<const float4 *>(vnew_t)[dq];
                o[0] = fmaf(wn, vn.x, o[0]);
                o[1] = fmaf(wn, vn.y, o[1]);
                o[2] = fmaf(wn, vn.z, o[2]);
                o[3] = fmaf(wn, vn.w, o[3]);
            }
            store_out(h, dq, o);
        }
        if (threadIdx.x < G) a.lse[qrow(threadIdx.x)] = lse_s[threadIdx.x];
        store_new_entries();
        return;
    }

    // This chunk's partial: kept in shared memory (a multi-token pass with one
    // chunk combines from it) and, when the sequence has several chunks, written out.
    for (int i = threadIdx.x; i < G * (kHeadDim / 4); i += blockDim.x) {
        const int h = i / (kHeadDim / 4), dq = i % (kHeadDim / 4);
        const float4 o4 = warp_sum(h, dq);
        reinterpret_cast<float4 *>(own_o)[i] = o4;
        if (nchunks > 1)
            __stcg(reinterpret_cast<float4 *>(a.part_o) + (pbase + (size_t)h * a.max_chunks + chunk) * (kHeadDim / 4) + dq,
                   o4);
    }
    if (nchunks > 1 && threadIdx.x < G)
        __stcg(a.part_ml + pbase + (size_t)threadIdx.x * a.max_chunks + chunk, own_ml[threadIdx.x]);
    __syncthreads();

    // Ticket: the last chunk of this (sequence, kv head) to finish does the combine.
    // The acq_rel atomic publishes this CTA's partial (ordered after the barrier)
    // and, for the last CTA, makes every other chunk's partial visible.
    if (nchunks > 1) {
        if (threadIdx.x == 0) {
            int *ctr = a.counters + (size_t)b * a.num_kv_heads + kvh;
            int ticket;
            asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(ticket) : "l"(ctr) : "memory");
            const int last = ticket == nchunks - 1;
            if (last) atomicExch(ctr, 0);  // ready for the next call on this stream
            *flag_s = last;
        }
        __syncthreads();
        if (!*flag_s) return;
    }

    // ---- combine (one CTA per sequence and kv head) ----
    // A single-token pass made its new entry, its scores, sink and gate values
    // in the prologue; a multi-token pass reads and makes them here, with each
    // warp's chunk maxima and sums requested in the same round.
    if (MT && threadIdx.x < G) {   // per row: the sink of its head, the gate logit of its token and head
        sink_s[threadIdx.x] = a.sink ? a.sink[kvh * Gm + threadIdx.x % Gm] : 0.f;
        gate_s[threadIdx.x] = a.gate ? a.gate[qrow(threadIdx.x)] : 0.f;
    }
    const float2 *pml = reinterpret_cast<const float2 *>(a.part_ml);
    constexpr int kPerLane = 4;
    float2 ml[kPerLane];
    {
        const int h = warp < G ? warp : 0;
        const size_t ph = pbase + (size_t)h * a.max_chunks;
#pragma unroll
        for (int r = 0; r < kPerLane; ++r) {
            const int j = lane + 32 * r;
            ml[r] = make_float2(-INFINITY, 0.f);
            if (j < nchunks) ml[r] = nchunks == 1 ? own_ml[h] : __ldcg(pml + ph + j);
        }
    }
    // New entries made here: a multi-token pass's, or a step grid's longer sequence's.
    const bool new_late = has_new && !new_early;
    if (!MT && new_late && (int)threadIdx.x < (codes_ld ? 32 : 64)) {
        const int per = codes_ld ? 16 : 32, t = threadIdx.x;
        const size_t e = ((size_t)b * a.num_kv_heads + kvh) * kHeadDim * (codes_ld ? 1 : 2);
        const uint4 x = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(t < per ? a.new_k : a.new_v) + e)[t % per];
        if (codes_ld) {
            reinterpret_cast<uint4 *>(code_s + (t < per ? 0 : kHeadDim))[t % per] = x;
        } else {
            float f[8];
            unpack_bf16x8(x, f);
            float4 *dst = reinterpret_cast<float4 *>((t < per ? kraw_s : vnew_s) + (t % per) * 8);
            dst[0] = make_float4(f[0], f[1], f[2], f[3]);
            dst[1] = make_float4(f[4], f[5], f[6], f[7]);
        }
    }
    if (new_late) {
        __syncthreads();
        make_new_entries();
    }
    __syncthreads();
    // Per row: M = max(chunk maxima, new scores), chunk weights 2^(m_j - M) and
    // L = sum of weighted chunk sums (+ the new entries).  Warp w takes rows w, w + warps, ...
    float *wts = reinterpret_cast<float *>(smem);   // [G][nchunks] (the warp buffers are free)
    for (int h = warp; h < G; h += kNThreads / 32) {
        const size_t ph = pbase + (size_t)h * a.max_chunks;
        if (h != warp) {  // a second row for this warp: its pairs were not preloaded
#pragma unroll
            for (int r = 0; r < kPerLane; ++r) {
                const int j = lane + 32 * r;
                ml[r] = make_float2(-INFINITY, 0.f);
                if (j < nchunks) ml[r] = nchunks == 1 ? own_ml[h] : __ldcg(pml + ph + j);
            }
        }
        // Scores of the new entries row h sees: its own token's and (MT) the earlier tokens'.
        const int th = MT ? h / Gm : 0;
        float s_new = -INFINITY;
        if (has_new) {
            if (!new_late) {
                s_new = wnew_t[h];   // scored in the prologue
            } else {
                for (int j = 0; j <= th; ++j) {
                    float t = 0.f;
                    for (int d = lane; d < kHeadDim; d += 32) {
                        float qv;
                        if constexpr (kUmma) {   // the q operand: bf16 high and low parts
                            const uint16_t *q16 = reinterpret_cast<const uint16_t *>(q_s);
                            qv = __uint_as_float((uint32_t)q16[umma_q_offset<G>(h, d) / 2] << 16) +
                                 __uint_as_float((uint32_t)q16[umma_q_offset<G>(G + h, d) / 2] << 16);
                        } else {
                            qv = q_join<KV>(q_w[h * kHeadDim + d]);
                        }
                        t = fmaf(qv, knew_t[j * kHeadDim + d], t);
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
                    if (lane == 0) wnew_t[h * WN + j] = t;
                    s_new = fmaxf(s_new, t);
                }
            }
            __syncwarp();
        }
        float M = s_new;
#pragma unroll
        for (int r = 0; r < kPerLane; ++r) M = fmaxf(M, ml[r].x);
        for (int j = lane + 32 * kPerLane; j < nchunks; j += 32) M = fmaxf(M, __ldcg(pml + ph + j).x);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float L = 0.f;
#pragma unroll
        for (int r = 0; r < kPerLane; ++r) {
            const int j = lane + 32 * r;
            if (j < nchunks) {
                const float w = (ml[r].x == -INFINITY) ? 0.f : fast_exp2(ml[r].x - M);
                wts[h * nchunks + j] = w;
                L = fmaf(w, ml[r].y, L);
            }
        }
        for (int j = lane + 32 * kPerLane; j < nchunks; j += 32) {
            const float2 m2 = __ldcg(pml + ph + j);
            const float w = (m2.x == -INFINITY) ? 0.f : fast_exp2(m2.x - M);
            wts[h * nchunks + j] = w;
            L = fmaf(w, m2.y, L);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
        float w_new = 0.f;   // lane j <= th: weight of new entry j
        if (has_new && lane <= th) w_new = fast_exp2(wnew_t[h * WN + lane] - M);
        __syncwarp();
        if (has_new && lane <= th) wnew_t[h * WN + lane] = w_new;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) w_new += __shfl_xor_sync(0xffffffffu, w_new, off);
        L += w_new;
        if (lane == 0) {
            const float lse = (M + fast_log2(L)) * kLn2;
            float f = a.sink ? 1.f / (1.f + fast_exp2((sink_s[h] - lse) * kLog2e)) : 1.f;
            if (a.gate) f *= 1.f / (1.f + fast_exp2(-gate_s[h] * kLog2e));
            head_s[h] = f / L * vscale;   // FP8: partials and the new value are in V-code units
            a.lse[qrow(h)] = lse;
        }
    }
    __syncthreads();
    // Outputs: thread t < 128 owns dims [4*(t%64), +4) of every row for the
    // chunks of parity t/64, several chunks' loads in flight at once; the two
    // parities meet in shared memory.
    float4 *half_s = reinterpret_cast<float4 *>(wts + ((G * nchunks + 3) & ~3));   // [G][64], 16-byte aligned
    const int dq = threadIdx.x & 63, parity = threadIdx.x >> 6;
    float4 acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (nchunks == 1) {
        if (parity == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float4 v = reinterpret_cast<const float4 *>(own_o)[h * 64 + dq];
                const float w = wts[h];
                acc[h] = make_float4(w * v.x, w * v.y, w * v.z, w * v.w);
            }
        }
    } else if (parity < 2) {
        const float4 *po = reinterpret_cast<const float4 *>(a.part_o) + pbase * (kHeadDim / 4) + dq;
        constexpr int U = G >= 16 ? 1 : (G >= 8 ? 2 : 4);   // chunks per round of loads
        int j = parity;
        for (; j + 2 * (U - 1) < nchunks; j += 2 * U) {
            float4 v[U][G];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int h = 0; h < G; ++h) v[u][h] = __ldcg(po + ((size_t)h * a.max_chunks + j + 2 * u) * (kHeadDim / 4));
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float w = wts[h * nchunks + j + 2 * u];
                    acc[h].x = fmaf(w, v[u][h].x, acc[h].x);
                    acc[h].y = fmaf(w, v[u][h].y, acc[h].y);
                    acc[h].z = fmaf(w, v[u][h].z, acc[h].z);
                    acc[h].w = fmaf(w, v[u][h].w, acc[h].w);
                }
        }
        for (; j < nchunks; j += 2) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float w = wts[h * nchunks + j];
                const float4 v = __ldcg(po + ((size_t)h * a.max_chunks + j) * (kHeadDim / 4));
                acc[h].x = fmaf(w, v.x, acc[h].x);
                acc[h].y = fmaf(w, v.y, acc[h].y);
                acc[h].z = fmaf(w, v.z, acc[h].z);
                acc[h].w = fmaf(w, v.w, acc[h].w);
            }
        }
    }
    if (parity == 1) {
#pragma unroll
        for (int h = 0; h < G; ++h) half_s[h * 64 + dq] = acc[h];
    }
    __syncthreads();
    if (parity == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float4 o1 = half_s[h * 64 + dq];
            float o[4] = {acc[h].x + o1.x, acc[h].y + o1.y, acc[h].z + o1.z, acc[h].w + o1.w};
            if (has_new) {
                const int th = MT ? h / Gm : 0;
                for (int j = 0; j <= th; ++j) {
                    const float wn = wnew_t[h * WN + j];
                    const float4 vn = *reinterpret_cast<const float4 *>(vnew_t + j * kHeadDim + 4 * dq);
                    o[0] = fmaf(wn, vn.x, o[0]);
                    o[1] = fmaf(wn, vn.y, o[1]);
                    o[2] = fmaf(wn, vn.z, o[2]);
                    o[3] = fmaf(wn, vn.w, o[3]);
                }
            }
            store_out(h, dq, o);
        }
    }
    store_new_entries();
}

template <int G, int CONSUMER, int S, int KV, bool MT, int NL>
cudaError_t launch_g(const LaunchTable<NL> &p, dim3 grid, bool pdl, cudaStream_t s) {
    static std::atomic<uint64_t> configured{0};   // devices whose attribute is set
    const size_t smem = layer_smem_bytes(G, S * kv_stage_bytes(KV) / kStageBytes) +
                        (umma_pass(G, KV, MT, deep_ring(S, KV), CONSUMER) ? umma_extra_bytes(G) : 0);
    int device = -1;
    if (!done_on_device(configured, &device)) {
        cudaError_t e = cudaFuncSetAttribute(attn_layer_kernel<G, CONSUMER, S, KV, MT, NL>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess && NL == 1)   // clusters of up to 16 CTAs (single-layer launches)
            e = cudaFuncSetAttribute(attn_layer_kernel<G, CONSUMER, S, KV, MT, NL>,
                                     cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        mark_done_on_device(configured, device);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(layer_threads(G, KV, NL, MT, deep_ring(S, KV), CONSUMER));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n++].val.programmaticStreamSerializationAllowed = 1;
    }
    if (NL == 1 && p.layer[0].a.cluster > 1) {
        if (MT || S * kv_stage_bytes(KV) <= kStages * kStageBytes || grid.x != (unsigned)p.layer[0].a.cluster ||
            p.layer[0].a.cluster > kMaxCluster)
            return cudaErrorInvalidValue;
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)p.layer[0].a.cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n++].val.clusterDim.z = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, attn_layer_kernel<G, CONSUMER, S, KV, MT, NL>, p);
}

// Largest cluster size (16, then 8) with which the single-layer deep-ring kernel
// (tensor-core consumer, one token) fits at least one cluster on the device; 0 if
// neither does.
template <int G, int KV>
int cluster_limit_g() {
    constexpr int S = kDeepStages * kStageBytes / kv_stage_bytes(KV);
    auto kernel = attn_layer_kernel<G, CONSUMER_MMA, S, KV, false, 1>;
    const size_t smem = layer_smem_bytes(G, kDeepStages);
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
        cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return 0;
    for (int k : {kMaxCluster, 8}) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(k, 1, 1);
        cfg.blockDim = dim3(layer_threads(G, KV, 1, false, true));
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)k;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) == cudaSuccess && clusters > 0) return k;
        cudaGetLastError();   // clear a refused query
    }
    return 0;
}

// S counts stages of the cache's type: an E4M3 ring has twice the bf16 count.
// rows: query rows per kv head (group x tokens of the pass); mt: a pass of a
// multi-token step.  Step tables (NL > 1) run the tensor-core consumer only.
template <int CONSUMER, int S_BF16, int KV, int NL>
cudaError_t launch_c(const LaunchTable<NL> &p, dim3 grid, int rows, bool mt, bool pdl, cudaStream_t s) {
    constexpr int S = S_BF16 * kStageBytes / kv_stage_bytes(KV);
    if (mt) {   // tensor-core consumer, rows = group x tokens
        if (CONSUMER != CONSUMER_MMA) return cudaErrorInvalidValue;
        switch (rows) {
        case 1: return launch_g<1, CONSUMER_MMA, S, KV, true, NL>(p, grid, pdl, s);
        case 2: return launch_g<2, CONSUMER_MMA, S, KV, true, NL>(p, grid, pdl, s);
        case 4: return launch_g<4, CONSUMER_MMA, S, KV, true, NL>(p, grid, pdl, s);
        case 8: return launch_g<8, CONSUMER_MMA, S, KV, true, NL>(p, grid, pdl, s);
        case 16:   // 16 rows: one CTA per SM with the deep ring
            if constexpr (S_BF16 == kDeepStages) return launch_g<16, CONSUMER_MMA, S, KV, true, NL>(p, grid, pdl, s);
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
        }
    }
    switch (rows) {
    case 1: return launch_g<1, CONSUMER, S, KV, false, NL>(p, grid, pdl, s);
    case 2: return launch_g<2, CONSUMER, S, KV, false, NL>(p, grid, pdl, s);
    case 4: return launch_g<4, CONSUMER, S, KV, false, NL>(p, grid, pdl, s);
    case 8: return launch_g<8, CONSUMER, S, KV, false, NL>(p, grid, pdl, s);
    default: return cudaErrorInvalidValue;
    }
}

template <int KV, int NL>
cudaError_t launch_kv(const LaunchTable<NL> &p, dim3 grid, int rows, bool mt, int consumer, int stages, bool pdl,
                      cudaStream_t s) {
    // Multi-token passes of 32 rows over bf16 caches (more than mma.sync holds in
    // registers) run the tcgen05 pass with a 128 KiB ring; with the tensor-memory
    // consumer so do 16-row passes.  Every other pass runs mma.sync.
    if (consumer == CONSUMER_UMMA || consumer == CONSUMER_MMA) {
        if constexpr (KV == KV_BF16) {
            if (consumer == CONSUMER_UMMA && mt && rows == 16 && stages == kDeepStages)
                return launch_g<16, CONSUMER_UMMA, kDeepStages, KV_BF16, true, NL>(p, grid, pdl, s);
            if (mt && rows == 32 && stages == kUmma32Stages)   // three K-half and two V-half slots
                return launch_g<32, CONSUMER_UMMA, kUmma32Stages, KV_BF16, true, NL>(p, grid, pdl, s);
        }
        if (rows > kMaxRowsMma) return cudaErrorInvalidValue;
        consumer = CONSUMER_MMA;
    }
    if constexpr (NL > 1) {
        if (consumer != CONSUMER_MMA) return cudaErrorInvalidValue;
        if constexpr (KV == KV_FP8) {   // three CTAs per SM: single-token grids of kTripleRows rows
            if (stages == kTripleStages) {
                if (mt || rows != kTripleRows) return cudaErrorInvalidValue;
                return launch_g<kTripleRows, CONSUMER_MMA, kTripleStages, KV, false, NL>(p, grid, pdl, s);
            }
        }
        return stages == kDeepStages ? launch_c<CONSUMER_MMA, kDeepStages, KV, NL>(p, grid, rows, mt, pdl, s)
                                     : launch_c<CONSUMER_MMA, kStages, KV, NL>(p, grid, rows, mt, pdl, s);
    } else {
        if (stages == kDeepStages)
            return consumer == CONSUMER_MMA ? launch_c<CONSUMER_MMA, kDeepStages, KV, NL>(p, grid, rows, mt, pdl, s)
                                            : launch_c<CONSUMER_FMA, kDeepStages, KV, NL>(p, grid, rows, mt, pdl, s);
        return consumer == CONSUMER_MMA ? launch_c<CONSUMER_MMA, kStages, KV, NL>(p, grid, rows, mt, pdl, s)
                                        : launch_c<CONSUMER_FMA, kStages, KV, NL>(p, grid, rows, mt, pdl, s);
    }
}

}  // namespace
}  // namespace hd
