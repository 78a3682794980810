// Internal declarations shared by the host API and the CUDA kernels of the
// hybrid decode-attention library.  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "hybrid_decode.h"

namespace hd {

constexpr int kHeadDim = 256;     // head_dim this build implements
constexpr int kMaxGroup = 8;      // query heads per kv head
constexpr int kStageKeys = 32;    // keys per pipeline stage (rows of one TMA box)
constexpr int kStages = 3;        // stages in flight per CTA
constexpr int kBoxCols = 64;      // bf16 columns per 128-byte swizzled box row
constexpr int kBoxesPerRow = kHeadDim / kBoxCols;                 // 4
constexpr int kBoxBytes = kStageKeys * 128;                       // 4 KiB
constexpr int kStageBytes = 2 * kBoxesPerRow * kBoxBytes;         // K + V: 32 KiB
constexpr int kChunkMin = 64;
constexpr int kChunkMax = 512;

// Which keys a split CTA scores for sequence b with c = context[b] previous tokens.
enum KeySet : int32_t {
    KEYS_RING = 0,  // cached ring slots [0, min(c, capacity)); the new entry is scored by the combine
    KEYS_ROLL = 1,  // rolled window [0, min(c + 1, window)) (the new entry is already in it)
    KEYS_FULL = 2   // positions [0, c] (the new entry was appended at index c)
};

// Split-K pass: one CTA per (chunk, kv head, sequence).
struct SplitArgs {
    const int32_t *context;
    const float *q_rot;      // [batch][Hq][D]
    float *part_o;           // [batch][Hq][max_chunks][D] unnormalised partial outputs
    float2 *part_ml;         // [batch][Hq][max_chunks] (running max in log2 units, sum)
    int32_t *err;
    int32_t num_q_heads, num_kv_heads;
    int32_t chunk_keys, max_chunks;
    int32_t key_set, capacity, window, max_context;
};

// LSE combine + sink + ring commit: one CTA per (kv head, sequence).
struct CombineArgs {
    const int32_t *context;
    const float *q_rot;
    const float *part_o;
    const float2 *part_ml;
    const float *sink;                 // [Hq] or null
    __nv_bfloat16 *out;                // [batch][Hq][D]
    float *lse;                        // [batch][Hq]
    const __nv_bfloat16 *stage_k;      // ring staging [batch][Hkv][D] (KEYS_RING only)
    const __nv_bfloat16 *stage_v;
    __nv_bfloat16 *cache_k;            // ring commit target (KEYS_RING only)
    __nv_bfloat16 *cache_v;
    int64_t seq_stride;
    int32_t capacity;
    int32_t *err;
    int32_t num_q_heads, num_kv_heads;
    int32_t chunk_keys, max_chunks;
    int32_t key_set, window, max_context;
};

// Partial RoPE of q and the new k, and the K/V store.
struct RopeArgs {
    const int32_t *context;
    const __nv_bfloat16 *q;            // [batch][Hq][D]
    const __nv_bfloat16 *k;            // [batch][Hkv][D]
    const __nv_bfloat16 *v;
    float *q_rot;                      // [batch][Hq][D]
    const float2 *table;               // [max_context + 1][rotary_dim / 2] (cos, sin)
    __nv_bfloat16 *dst_k;              // full: cache; ring: staging; roll: cache
    __nv_bfloat16 *dst_v;
    int64_t seq_stride;                // of dst (staging: Hkv * D)
    int32_t capacity;                  // of dst (staging: 1)
    int32_t *err;
    int32_t num_q_heads, num_kv_heads, rotary_dim;
    int32_t key_set, window, max_context;
};

cudaError_t launch_rope_append(const RopeArgs &a, int batch, cudaStream_t s);
cudaError_t launch_roll_window(const RopeArgs &a, int batch, cudaStream_t s);
cudaError_t launch_split(const CUtensorMap *kmap, const CUtensorMap *vmap, const SplitArgs &a,
                         int batch, int group, cudaStream_t s);
cudaError_t launch_combine(const CombineArgs &a, int batch, int group, cudaStream_t s);
size_t split_smem_bytes();

}  // namespace hd
