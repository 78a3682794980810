// Internal declarations shared by the host API and the CUDA kernels of the
// hybrid decode-attention library.  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <type_traits>

#include "hybrid_decode.h"

// Build switches shared by the host planner and the kernels (measured choices).
// 16-row multi-token passes over bf16 caches take 64-key stages (two 8-row
// groups, 16 keys per consumer warp and call).
#ifndef HD_WIDE_MT
#define HD_WIDE_MT 1
#endif
// The 64-key stages of those passes (and of the tcgen05 passes) load one 64-row
// box per 128-byte column of K and V -- 8 copies a stage -- instead of two
// 32-row boxes.
#ifndef HD_WIDE_BOX64
#define HD_WIDE_BOX64 1
#endif

namespace hd {

// Per-device one-time setup (kernel attributes are set per device): true when
// `done` already has the current device's bit; otherwise the caller does the
// setup and then calls mark_done_on_device.  Devices past 63 always redo it.
inline bool done_on_device(const std::atomic<uint64_t> &done, int *device) {
    if (cudaGetDevice(device) != cudaSuccess) *device = -1;
    return *device >= 0 && *device < 64 && (done.load(std::memory_order_acquire) >> *device & 1u);
}
inline void mark_done_on_device(std::atomic<uint64_t> &done, int device) {
    if (device >= 0 && device < 64) done.fetch_or(1ull << device, std::memory_order_release);
}

constexpr int kHeadDim = 256;     // the head_dim this library implements
constexpr int kMaxGroup = 8;      // query heads per kv head
constexpr int kStageKeys = 32;    // keys per pipeline stage (rows of one TMA box)
constexpr int kStages = 3;        // bf16 stages per CTA with two CTAs per SM (the default)
constexpr int kDeepStages = 6;    // bf16 stages per CTA with one CTA per SM (grids of at most one CTA per SM)
constexpr int kTripleStages = 2;  // stages per CTA with three CTAs per SM (E4M3 step grids of 4 rows)
constexpr int kTripleRows = 4;
constexpr int kBoxCols = 64;      // bf16 columns per 128-byte swizzled box row
constexpr int kBoxesPerRow = kHeadDim / kBoxCols;                 // 4
constexpr int kBoxBytes = kStageKeys * 128;                       // 4 KiB
constexpr int kStageBytes = 2 * kBoxesPerRow * kBoxBytes;         // K + V: 32 KiB

// Cache element types (hd_kv_dtype).  A stage is 32 KiB of K + V either way:
// 32 bf16 keys (four 64-column boxes per row block) or 64 E4M3 keys (two
// 128-column boxes of 64 rows), so both rings have the same stage counts.
enum KvType : int32_t { KV_BF16 = 0, KV_FP8 = 1 };
__host__ __device__ constexpr int kv_elem_bytes(int kv) { return kv == KV_FP8 ? 1 : 2; }
__host__ __device__ constexpr int kv_stage_keys(int kv) { return kv == KV_FP8 ? 64 : kStageKeys; }   // box rows
__host__ __device__ constexpr int kv_box_cols(int kv) { return 128 / kv_elem_bytes(kv); }            // 64 / 128
__host__ __device__ constexpr int kv_boxes_per_row(int kv) { return kHeadDim * kv_elem_bytes(kv) / 128; }  // 4 / 2
__host__ __device__ constexpr int kv_box_bytes(int kv) { return kv_stage_keys(kv) * 128; }            // 4 / 8 KiB
__host__ __device__ constexpr int kv_stage_bytes(int kv) { return 2 * kv_boxes_per_row(kv) * kv_box_bytes(kv); }
static_assert(kv_stage_bytes(KV_BF16) == kStageBytes && kv_stage_bytes(KV_FP8) == kStageBytes,
              "both cache types use 32 KiB stages");
constexpr int kMaxTokens = 8;     // tokens per sequence of one multi-token step
constexpr int kMaxRows = 32;      // query rows per kv head in one kernel (heads x tokens)
constexpr int kMaxRowsMma = 16;   // ... with the mma.sync consumers (32: the tcgen05 pass only)
// Shared-memory bytes the multi-token combine keeps at the end of the ring: new
// K/V values and codes, per-row new-entry weights, and per-row sink, gate and scale.
constexpr int kMtNewBytes =
    2 * kMaxTokens * kHeadDim * 4 + 2 * kMaxTokens * kHeadDim + kMaxRows * kMaxTokens * 4 + 3 * kMaxRows * 4;
constexpr int kChunkMin = 64;
constexpr int kChunkMax = 2048;

// Split plan: keys per chunk (a power of two from kChunkMin to kChunkMax) and
// chunks per sequence for `max_keys` keys, keeping batch * chunks <= max_slots.
// chunk_max: kChunkMax for bf16 caches; E4M3 caches use twice as many keys per
// chunk (the same bytes per CTA), which measured 10 % faster at 131k contexts.
void plan_split(int64_t batch, int64_t num_kv_heads, int64_t max_keys, int64_t num_sms,
                int64_t max_slots, int32_t *chunk_keys, int32_t *num_chunks, int32_t *stages = nullptr,
                int64_t chunk_max = kChunkMax);

// bf16 stages of the one-CTA-per-SM ring for a pass of more than kMaxGroup rows:
// the 32-row tensor-memory pass keeps 160 KiB -- three K halves and two V halves of
// 64-key stages (its q operand takes 32 KiB).
constexpr int kUmma32Stages = 5;
inline int deep_stages_for(size_t rows) { return rows > (size_t)kMaxRowsMma ? kUmma32Stages : kDeepStages; }

// Passes of 64-key bf16 stages: 16 rows on mma.sync (HD_WIDE_MT) or on tcgen05,
// and 32 rows (tcgen05 only).  Their tensor maps have kWideBoxRows-row boxes.
constexpr int kWideBoxRows = HD_WIDE_BOX64 ? 2 * kStageKeys : kStageKeys;
inline bool wide_stage_pass(int kv, size_t rows, bool tensor_memory) {
    return kv == KV_BF16 && rows > (size_t)kMaxGroup && (HD_WIDE_MT || tensor_memory || rows > (size_t)kMaxRowsMma);
}

// Ring of a step grid with more CTAs than SMs.  Single-token E4M3 grids of
// kTripleRows rows (group 4) run three CTAs per SM on two-stage rings: twelve
// consumer warps per SM hide more of the per-tile conversion and MMA chain than
// eight do on three-stage rings (the batch-64 E4M3 step 1.206 -> 1.175 ms, the
// 131k-context one 0.543 -> 0.536 ms).  At the 168 registers that three CTAs
// leave a thread, groups 1 and 2 spill, and group 8 does not fit three rings in
// shared memory; those grids, and all others, keep two CTAs per SM.
inline int step_stages(int kv, size_t rows, bool mt) {
    if (rows > (size_t)kMaxGroup) return deep_stages_for(rows);
    return kv == KV_FP8 && !mt && rows == (size_t)kTripleRows ? kTripleStages : kStages;
}

// Shared memory of the combine: a weight per (query row, chunk) plus a float4
// row per query row (and, for a multi-token pass, the new entries), inside the
// stage ring of `stages` bf16 stages that the CTA no longer needs then.
inline bool combine_fits(size_t rows, int64_t num_chunks, bool mt, int stages) {
    return (rows * num_chunks + 3) * sizeof(float) + rows * 64 * 16 + (mt ? kMtNewBytes : 0) <=
           (size_t)stages * kStageBytes;
}

// Which cache rows the split pass scores for sequence b with c = context[b].
enum KeySet : int32_t {
    KEYS_RING = 0,         // ring slots [0, min(c, capacity)); the new entry is scored apart
    KEYS_ROLL = 1,         // rolled window [0, min(c + 1, window)), the new entry already in it
    KEYS_FULL_CACHED = 2,  // positions [0, c]: the new entry was appended at index c
    KEYS_FULL_PREV = 3,    // positions [0, c): the new entry is scored apart and appended
    KEYS_ROLL_SHIFT = 4    // rolled window before this pass's shift: rows [0, c) while it is not
                           // full, else rows [1, window) (row 0 leaves the window); the new entries
                           // are scored apart, the kernel shifts the rows it read down by
                           // sh = max(0, min(c, window) + tokens - window) rows and stores token t's
                           // entry at row min(c, window) + t - sh; one chunk per sequence
};
// Where the new entry comes from when it is scored apart from the cache.
enum NewEntry : int32_t {
    NEW_NONE = 0,     // already in the scored cache rows
    NEW_ROTATE = 1,   // bf16 k of the step, rotated (fp64, one rounding) in the kernel
    NEW_STAGED = 2    // already rotated and rounded (ring staging row, in the cache's type)
};
// Where the new entry is stored once every chunk has read the cache.
enum Commit : int32_t { COMMIT_NONE = 0, COMMIT_APPEND = 1, COMMIT_RING = 2, COMMIT_ROLL = 3 };
enum Consumer : int32_t { CONSUMER_FMA = 0, CONSUMER_MMA = 1, CONSUMER_UMMA = 2 };
// Tensor-core consumers (mma.sync, or tcgen05 for the passes it takes).
constexpr bool tensor_consumer(int c) { return c == CONSUMER_MMA || c == CONSUMER_UMMA; }

// One attention layer: one CTA per (chunk, kv head, sequence); the last CTA of
// each (sequence, kv head) combines the chunks.
struct LayerArgs {
    const int32_t *context;
    const __nv_bfloat16 *q_bf16;   // [batch][Hq][D], rotated in the kernel ...
    const float *q_rot;            // ... or already rotated, fp32 (when q_bf16 is null)
    const float2 *table;           // [max_context + 1][rotary_dim / 2] (cos, sin)
    int32_t rotary_dim;
    const void *new_k;             // [batch][Hkv][D] (NEW_ROTATE: raw bf16 k; NEW_STAGED: staged entry)
    const void *new_v;
    int32_t new_kind, commit, key_set;
    void *cache_k;                 // cache of the layer (also the store target), bf16 or E4M3 codes
    void *cache_v;
    int64_t seq_stride;            // elements
    int32_t capacity;
    int32_t kv_type;               // KV_BF16 / KV_FP8
    const float *k_scale;          // FP8: [Hkv] dequantisation scales, else null
    const float *v_scale;
    const float *sink;             // [Hq] or null
    const float *gate;             // [batch][Hq] output-gate logits or null
    __nv_bfloat16 *out;            // [batch][Hq][D]
    float *lse;                    // [batch][Hq]
    float *part_o;                 // [batch][Hq][max_chunks][D] unnormalised partial outputs
    float2 *part_ml;               // [batch][Hq][max_chunks] (max in log2 units, sum)
    int32_t *counters;             // [max_batch][Hkv], zero between calls
    int32_t *err;
    int32_t num_q_heads, num_kv_heads;
    int32_t chunk_keys, max_chunks;
    int32_t window, max_context;
    int32_t drop_stage;            // test hook: producers stop issuing at this stage (-1: off)
    // Multi-token decode: this launch takes `tokens` tokens (1: the single-token
    // step) of `total_tokens` per sequence, starting at token `token0`, at
    // positions context + token0 + t; q/k/v/out/lse/gate then carry a token index
    // after the batch index.
    int32_t tokens, token0, total_tokens;
    // Single-layer launches only: > 1 when the grid runs in thread-block clusters of
    // that many CTAs along the chunk dimension (every chunk of a (sequence, kv head)
    // in one cluster), whose partials then merge through distributed shared memory.
    int32_t cluster;
    // Launched as a programmatic dependent in full stream order: the kernel waits
    // for the previous grid before its first read (0: only before its first write).
    int32_t wait_first;
};

// Partial RoPE of q and the new k, and the K/V store.
struct RopeArgs {
    const int32_t *context;
    const __nv_bfloat16 *q;            // [batch][Hq][D]
    const __nv_bfloat16 *k;            // [batch][Hkv][D]
    const __nv_bfloat16 *v;
    float *q_rot;                      // [batch][Hq][D]
    const float2 *table;               // [max_context + 1][rotary_dim / 2] (cos, sin)
    void *dst_k;                       // full: cache; ring: staging; roll: cache (bf16 or E4M3)
    void *dst_v;
    int64_t seq_stride;                // of dst, elements (staging: Hkv * D)
    int32_t capacity;                  // of dst (staging: 1)
    int32_t kv_type;                   // KV_BF16 / KV_FP8
    const float *k_scale;              // FP8: [Hkv] scales, else null
    const float *v_scale;
    int32_t *err;
    int32_t num_q_heads, num_kv_heads, rotary_dim;
    int32_t key_set, window, max_context;
};

// Kernel parameters of an attention launch: a table of layers, each with its
// K and V cache views and arguments.  A single-layer launch (NL = 1) runs a
// (chunks, kv heads, sequences) grid; a step table (NL = kStepLayers) runs a
// 1-D grid where layer i owns the CTAs [begin[i], begin[i + 1]), ordered
// (sequence, kv head, chunk) with the chunk fastest.  The range starts sit
// together at the front of the table, so a CTA finds its layer with one load
// per lane from one 128-byte line.
constexpr int kStepLayers = 32;
struct alignas(64) LayerLaunch {
    CUtensorMap kmap, vmap;
    LayerArgs a;
};
template <int NL>
struct LaunchTable {
    int32_t begin[NL];
    int32_t num_layers;
    LayerLaunch layer[NL];
};
using StepTable = LaunchTable<kStepLayers>;
static_assert(sizeof(StepTable) <= 32764, "kernel parameters are limited to 32764 bytes");

cudaError_t launch_rope_append(const RopeArgs &a, int batch, cudaStream_t s);
cudaError_t launch_roll_window(const RopeArgs &a, int batch, cudaStream_t s);
// `stages` in bf16 stages (kStages or kDeepStages); a.kv_type picks the kernel.
// pdl: launch as a programmatic dependent of the previous grid in the stream.
// Only correct when that grid is another layer kernel of the same step that
// writes nothing this launch reads before griddepcontrol.wait (its own inputs
// and its own cache): the kernel starts streaming before that grid is done.
cudaError_t launch_layer(const CUtensorMap *kmap, const CUtensorMap *vmap, const LayerArgs &a,
                         int batch, int group, int consumer, int stages, bool pdl, cudaStream_t s);
// One grid for the t.num_layers layers of a step table (num_ctas CTAs in all;
// every layer with the same cache type, rows per kv head and pass shape; a
// tensor-core consumer).  The layers must be independent: no layer reads or
// writes what another one writes.
cudaError_t launch_step(const StepTable &t, int num_ctas, int rows, bool mt, int kv, int consumer, int stages,
                        cudaStream_t s);
// Per-family launchers, one translation unit each (rows: query rows per kv
// head; mt: a pass of a multi-token step).
cudaError_t launch_layer_bf16(const LaunchTable<1> &t, dim3 grid, int rows, bool mt, int consumer, int stages,
                              bool pdl, cudaStream_t s);
cudaError_t launch_layer_fp8(const LaunchTable<1> &t, dim3 grid, int rows, bool mt, int consumer, int stages,
                             bool pdl, cudaStream_t s);
cudaError_t launch_step_bf16(const StepTable &t, dim3 grid, int rows, bool mt, int consumer, int stages,
                             cudaStream_t s);
cudaError_t launch_step_fp8(const StepTable &t, dim3 grid, int rows, bool mt, int stages, cudaStream_t s);
size_t layer_smem_bytes(int group, int stages);
// Largest cluster (16 or 8 CTAs, 0 if none) that single-layer launches of the
// deep-ring kernel for this group and cache type can run with on the current device.
int layer_cluster_limit(int group, int kv);
int layer_cluster_limit_fp8(int group);
constexpr int kMaxCluster = 16;

}  // namespace hd
