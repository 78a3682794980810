// Host side of the C ABI declared in include/hybrid_decode.h: argument
// validation, the context (RoPE tables, split-K workspace, ring staging rows),
// the split plan, TMA tensor maps and the kernel launches.
//
// The configuration checks mirror `SparkStepConfig.__post_init__` of
// vllm_omni/edge/spark_export.py (heads divisible by kv heads, known layer
// types, known cache layout); the sink checks mirror `_validate_sinks` of
// vllm/models/hy_v4/nvidia/flashmla_sparse.py (fp32 by type here, one value
// per query head, NULL for no sink).
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "hd_internal.h"

using namespace hd;

namespace hd {
// Chunk size of a step grid over `n` layers (batch[i] sequences of at most
// max_keys[i] scored keys; one_chunk[i]: the layer takes a single chunk of
// max(C, max_keys[i]) keys), with `rows` query rows per kv head and mt for a
// multi-token pass (the model is described at its definition below).
int32_t plan_step(int64_t num_kv_heads, int64_t num_sms, int kv_type, size_t rows, bool mt, int n,
                  const int32_t *batch, const int32_t *max_keys, const uint8_t *one_chunk);
}  // namespace hd

// Chunk size: the smallest power of two (64 .. chunk_max keys: 2048 bf16, 4096
// E4M3, i.e. the same bytes) that gives about
// one CTA per SM over the grid for the longest sequence bound.  If that grid
// fits in one CTA per SM, it runs so, with the deep ring (one CTA streams as
// much as two); otherwise the plan aims at two resident CTAs per SM with the
// default ring.  Short sliding layers get one or a few chunks per sequence;
// long full layers get long chunks (fewer per-CTA ramps, measured faster than
// filling whole waves with shorter ones); batch 1 gets many short chunks.
// Chunks grow further if the workspace bound requires it.
void hd::plan_split(int64_t batch, int64_t num_kv_heads, int64_t max_keys, int64_t num_sms,
                    int64_t max_slots, int32_t *chunk_keys, int32_t *num_chunks, int32_t *stages,
                    int64_t chunk_max) {
    auto chunks = [&](int64_t tt) { return max_keys > 0 ? (max_keys + tt - 1) / tt : 1; };
    auto pick = [&](int64_t target) {
        const int64_t want = (batch * num_kv_heads * max_keys + target - 1) / target;
        int64_t t = kChunkMin;
        while (t < want && t < chunk_max) t *= 2;
        while (t < chunk_max && batch * chunks(t) > max_slots) t *= 2;
        return t;
    };
    int64_t t = pick(num_sms);
    int32_t st = kDeepStages;
    if (batch * num_kv_heads * chunks(t) > num_sms) {
        t = pick(2 * num_sms);
        st = kStages;
    }
    *chunk_keys = (int32_t)t;
    *num_chunks = (int32_t)chunks(t);
    if (stages) *stages = st;
}

namespace {

struct MapCacheEntry {
    const void *k = nullptr, *v = nullptr;
    int64_t seq_stride = 0;
    int32_t capacity = 0, batch = 0;
    CUtensorMap kmap, vmap;     // boxes of one stage's keys
    bool wide_valid = false;    // kmapw / vmapw encoded for this cache
    CUtensorMap kmapw, vmapw;   // boxes of kWideBoxRows keys (64-key bf16 stages)
};

struct DeviceTable {
    float2 *data = nullptr;  // [max_context + 1][rotary_dim / 2]
    int32_t rotary_dim = 0;
};

struct LayerCall;

}  // namespace

struct hd_ctx {
    hd_config cfg;
    std::vector<int32_t> layer_types;
    int device = 0;
    int num_sms = 0;
    int group = 1;
    int sliding_layout = HD_LAYOUT_RING;
    DeviceTable table_sliding, table_full;
    float *part_o = nullptr;
    float2 *part_ml = nullptr;
    int64_t part_slots = 0;              // single-layer calls: capacity in (sequence, chunk) pairs
    int64_t part_rows = 0;               // capacity in partial rows ([256] floats + (m, l) each)
    uint8_t *stage_k = nullptr;          // [num_layers][max_batch][Hkv][D] entries of the cache type
    uint8_t *stage_v = nullptr;
    int kv_type = KV_BF16;
    int32_t *counters = nullptr;         // [num_layers][max_batch][Hkv] chunk tickets, zero between calls
    int32_t *err = nullptr;
    int consumer = CONSUMER_MMA;
    int cluster_max = 0;                 // largest cluster the single-layer kernel runs with (0: none)
    bool cluster_combine = true;         // single-layer calls: small grids merge chunks in a cluster
    int32_t drop_stage = -1;             // test hook, see hybrid_decode_inject_lost_copy
    bool layer_overlap = true;           // decode_step: layers start before the previous one finishes
    bool fuse_step = true;               // decode_step: one grid for all layers (step tables)
    StepTable step_table;                // parameters of the step grid being launched
    std::vector<LayerCall> step_calls;   // the layer calls of the step being launched
    std::vector<int> step_order;         // their order in the step grids
    // Last independence check of decode_step's layers (host memcmp of the array).
    std::vector<hd_layer_io> indep_layers;
    int32_t indep_batch = -1, indep_tokens = -1;
    bool indep_ok = false;
    int64_t launches = 0;
    std::vector<MapCacheEntry> maps;     // one per layer
    int32_t profile_mask = 0;           // bit (1 << layer type): bracket that type's launches
    bool profile_seen[2] = {false, false};  // FIRST_ONLY: a layer of that type was bracketed in this step
    std::vector<cudaEvent_t> ev_begin, ev_end;  // [3][kProfileEvents]: per layer type, then step grids
    size_t ev_used[3] = {0, 0, 0};
};

namespace {

constexpr int kProfileEvents = 4096;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int sliding_capacity(const hd_ctx *ctx) {
    return ctx->sliding_layout == HD_LAYOUT_ROLL ? ctx->cfg.sliding_window
                                                 : ctx->cfg.sliding_window - 1;
}

// Encodes the 4-D view {D, capacity, Hkv, batch} of one cache tensor with
// (128 bytes) x (box_rows keys) boxes and the 128-byte swizzle the consumers index by.
bool encode_cache_map(CUtensorMap *map, const void *base, int64_t seq_stride, int capacity,
                      int num_kv_heads, int batch, int kv_type, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t es = (cuuint64_t)kv_elem_bytes(kv_type);
    const cuuint64_t dims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)capacity,
                                (cuuint64_t)num_kv_heads, (cuuint64_t)batch};
    const cuuint64_t strides[3] = {(cuuint64_t)kHeadDim * es, (cuuint64_t)capacity * kHeadDim * es,
                                   (cuuint64_t)seq_stride * es};
    const cuuint32_t box[4] = {(cuuint32_t)kv_box_cols(kv_type), (cuuint32_t)box_rows, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, kv_type == KV_FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                    const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// wide: the maps of a pass of 64-key bf16 stages (wide_stage_pass).
hd_status maps_for(hd_ctx *ctx, int layer, const hd_kv_cache &c, int batch, bool wide, const CUtensorMap **km,
                   const CUtensorMap **vm) {
    MapCacheEntry &e = ctx->maps[layer];
    const int Hkv = ctx->cfg.num_kv_heads;
    if (e.k != c.k || e.v != c.v || e.seq_stride != c.seq_stride || e.capacity != c.capacity ||
        e.batch != batch) {
        const int rows = kv_stage_keys(ctx->kv_type);
        e.wide_valid = false;
        if (!encode_cache_map(&e.kmap, c.k, c.seq_stride, c.capacity, Hkv, batch, ctx->kv_type, rows) ||
            !encode_cache_map(&e.vmap, c.v, c.seq_stride, c.capacity, Hkv, batch, ctx->kv_type, rows)) {
            e.k = e.v = nullptr;
            return HD_ERR_CUDA;
        }
        e.k = c.k;
        e.v = c.v;
        e.seq_stride = c.seq_stride;
        e.capacity = c.capacity;
        e.batch = batch;
    }
    if (wide && !e.wide_valid) {
        if (!encode_cache_map(&e.kmapw, c.k, c.seq_stride, c.capacity, Hkv, batch, ctx->kv_type, kWideBoxRows) ||
            !encode_cache_map(&e.vmapw, c.v, c.seq_stride, c.capacity, Hkv, batch, ctx->kv_type, kWideBoxRows))
            return HD_ERR_CUDA;
        e.wide_valid = true;
    }
    *km = wide ? &e.kmapw : &e.kmap;
    *vm = wide ? &e.vmapw : &e.vmap;
    return HD_OK;
}

hd_status check_cache(const hd_ctx *ctx, const hd_kv_cache &c) {
    if (!c.k || !c.v || !aligned16(c.k) || !aligned16(c.v)) return HD_ERR_INVALID_ARG;
    if (c.capacity <= 0 || (c.seq_stride * kv_elem_bytes(ctx->kv_type)) % 16 != 0) return HD_ERR_INVALID_ARG;
    const bool fp8 = ctx->kv_type == KV_FP8;
    if (fp8 != (c.k_scale != nullptr) || fp8 != (c.v_scale != nullptr)) return HD_ERR_INVALID_ARG;
    if (c.seq_stride < (int64_t)ctx->cfg.num_kv_heads * c.capacity * kHeadDim)
        return HD_ERR_INVALID_ARG;
    return HD_OK;
}

// The context's workspace and tensor maps live on the device it was created on.
hd_status check_device(const hd_ctx *ctx) {
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess && dev == ctx->device ? HD_OK : HD_ERR_STATE;
}

hd_status check_call(const hd_ctx *ctx, int layer, int batch, const int32_t *context) {
    if (!ctx) return HD_ERR_INVALID_ARG;
    if (layer < 0 || layer >= ctx->cfg.num_layers) return HD_ERR_INVALID_ARG;
    if (batch <= 0 || !context) return HD_ERR_INVALID_ARG;
    if (batch > ctx->cfg.max_batch) return HD_ERR_CAPACITY;
    return HD_OK;
}

hd_status cuda_status(cudaError_t e) { return e == cudaSuccess ? HD_OK : HD_ERR_CUDA; }

// Workspace bound in (sequence, chunk) pairs: the largest chunk always fits
// (max_batch * ceil(max_keys / kChunkMax)); smaller chunks are allowed up to
// about two waves of CTAs on top of that.
int64_t part_slot_capacity(int max_batch, int max_keys, int num_sms) {
    return (int64_t)max_batch * ((max_keys + kChunkMax - 1) / kChunkMax) + 4LL * num_sms;
}

hd_status build_table(DeviceTable *t, int rotary_dim, double theta, int max_context) {
    const int half = rotary_dim / 2;
    t->rotary_dim = rotary_dim;
    if (half == 0) return HD_OK;
    std::vector<double> inv(half);
    for (int i = 0; i < half; ++i) inv[i] = 1.0 / std::pow(theta, (double)(2 * i) / rotary_dim);
    const size_t n = (size_t)(max_context + 1) * half;
    std::vector<float2> host(n);
    for (int64_t p = 0; p <= max_context; ++p)
        for (int i = 0; i < half; ++i) {
            const double ang = (double)p * inv[i];
            host[(size_t)p * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
        }
    if (cudaMalloc(&t->data, n * sizeof(float2)) != cudaSuccess) return HD_ERR_CUDA;
    if (cudaMemcpy(t->data, host.data(), n * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess)
        return HD_ERR_CUDA;
    return HD_OK;
}

void free_ctx(hd_ctx *ctx) {
    if (!ctx) return;
    cudaFree(ctx->table_sliding.data);
    cudaFree(ctx->table_full.data);
    cudaFree(ctx->part_o);
    cudaFree(ctx->part_ml);
    cudaFree(ctx->stage_k);
    cudaFree(ctx->stage_v);
    cudaFree(ctx->counters);
    cudaFree(ctx->err);
    for (auto e : ctx->ev_begin) cudaEventDestroy(e);
    for (auto e : ctx->ev_end) cudaEventDestroy(e);
    delete ctx;
}

// Launches the fused layer kernel (see attn_decode.cu) for one layer call.
struct LayerCall {
    int layer, batch;
    const int32_t *context;
    int max_keys;           // bound on the cached keys any sequence scores (split plan)
    int key_set, new_kind, commit;
    const void *q_bf16;     // rotate q in the kernel, or
    const float *q_rot;     // take it rotated
    const void *new_k, *new_v;
    hd_kv_cache cache;
    const float *sink;
    const float *gate;
    void *out;
    float *lse;
    bool pdl;               // previous grid in the stream is this step's previous layer kernel
    bool early = false;     // pdl: the layer may read and stream before that grid completes
    bool one_chunk = false; // step grids: the layer needs a single chunk per sequence
    int tokens = 1, token0 = 0, total_tokens = 1;   // multi-token decode: this pass's tokens
};

// Kernel arguments of one layer call with a given split; its partials start at
// partial row part_row0 of the workspace, its tickets at the layer's counters.
void fill_layer_args(const hd_ctx *ctx, const LayerCall &L, int32_t chunk_keys, int32_t num_chunks,
                     int64_t part_row0, LayerArgs &a) {
    const bool sliding = ctx->layer_types[L.layer] == HD_SLIDING;
    const DeviceTable &tab = sliding ? ctx->table_sliding : ctx->table_full;
    a = LayerArgs{};
    a.context = L.context;
    a.q_bf16 = static_cast<const __nv_bfloat16 *>(L.q_bf16);
    a.q_rot = L.q_rot;
    a.table = tab.data;
    a.rotary_dim = tab.rotary_dim;
    a.new_k = L.new_k;
    a.new_v = L.new_v;
    a.new_kind = L.new_kind;
    a.commit = L.commit;
    a.key_set = L.key_set;
    a.cache_k = L.cache.k;
    a.cache_v = L.cache.v;
    a.seq_stride = L.cache.seq_stride;
    a.capacity = L.cache.capacity;
    a.kv_type = ctx->kv_type;
    a.k_scale = L.cache.k_scale;
    a.v_scale = L.cache.v_scale;
    a.sink = L.sink;
    a.gate = L.gate;
    a.out = static_cast<__nv_bfloat16 *>(L.out);
    a.lse = L.lse;
    a.part_o = ctx->part_o + part_row0 * kHeadDim;
    a.part_ml = ctx->part_ml + part_row0;
    a.counters = ctx->counters + (size_t)L.layer * ctx->cfg.max_batch * ctx->cfg.num_kv_heads;
    a.err = ctx->err;
    a.num_q_heads = ctx->cfg.num_q_heads;
    a.num_kv_heads = ctx->cfg.num_kv_heads;
    a.chunk_keys = chunk_keys;
    a.max_chunks = num_chunks;
    a.window = ctx->cfg.sliding_window;
    a.max_context = ctx->cfg.max_context;
    a.drop_stage = ctx->drop_stage;
    a.tokens = L.tokens;
    a.token0 = L.token0;
    a.total_tokens = L.total_tokens;
    a.cluster = 0;
}

hd_status launch_layer_call(hd_ctx *ctx, const LayerCall &L, cudaStream_t stream) {
    const CUtensorMap *km = nullptr, *vm = nullptr;
    const bool wide = wide_stage_pass(ctx->kv_type, (size_t)ctx->group * L.tokens, ctx->consumer == CONSUMER_UMMA);
    hd_status st = maps_for(ctx, L.layer, L.cache, L.batch, wide, &km, &vm);
    if (st != HD_OK) return st;
    int32_t chunk_keys = 0, num_chunks = 0, stages = kStages;
    if (L.one_chunk) {   // a rolled window shifted in place: one CTA reads each sequence's window
        chunk_keys = (std::max(L.max_keys, 1) + kChunkMin - 1) / kChunkMin * kChunkMin;
        num_chunks = 1;
        stages = (int64_t)L.batch * ctx->cfg.num_kv_heads <= ctx->num_sms ? kDeepStages : kStages;
    } else {
        plan_split(L.batch, ctx->cfg.num_kv_heads, L.max_keys, ctx->num_sms, ctx->part_slots, &chunk_keys,
                   &num_chunks, &stages, ctx->kv_type == KV_FP8 ? 2 * kChunkMax : kChunkMax);
    }
    // Small grids (at most one CTA per SM) of single-token calls run every chunk
    // of a (sequence, kv head) in one thread-block cluster and merge the chunks'
    // partials in distributed shared memory, with no workspace round trip; the
    // sequence is then split into at most cluster_max chunks.
    int32_t cluster = 0;
    if (ctx->cluster_combine && ctx->cluster_max > 1 && L.total_tokens == 1 && !L.one_chunk && L.max_keys > 0) {
        const int64_t units = (int64_t)L.batch * ctx->cfg.num_kv_heads;
        int64_t ck = chunk_keys, k = num_chunks;
        if (k > ctx->cluster_max) {
            ck = ((L.max_keys + ctx->cluster_max - 1) / ctx->cluster_max + kChunkMin - 1) / kChunkMin * kChunkMin;
            k = (L.max_keys + ck - 1) / ck;
        }
        if (k > 1 && units * k <= ctx->num_sms) {
            chunk_keys = (int32_t)ck;
            num_chunks = (int32_t)k;
            stages = kDeepStages;
            cluster = (int32_t)k;
        }
    }
    if ((int64_t)ctx->group * L.tokens > kMaxGroup)   // 16 or 32 rows: one CTA per SM
        stages = deep_stages_for((size_t)ctx->group * L.tokens);
    if ((int64_t)L.batch * num_chunks > ctx->part_slots) return HD_ERR_CAPACITY;
    const size_t rows = (size_t)ctx->group * L.tokens;   // query rows per kv head
    if (!combine_fits(rows, num_chunks, L.total_tokens > 1, stages)) return HD_ERR_CAPACITY;
    LayerArgs a;
    fill_layer_args(ctx, L, chunk_keys, num_chunks, 0, a);
    a.cluster = cluster;
    a.wait_first = L.pdl && !L.early ? 1 : 0;

    const bool sliding = ctx->layer_types[L.layer] == HD_SLIDING;
    const int type = sliding ? HD_SLIDING : HD_FULL;
    const size_t slot = (size_t)type * kProfileEvents + ctx->ev_used[type];
    const bool timed = (ctx->profile_mask & (1 << type)) && ctx->ev_used[type] < (size_t)kProfileEvents &&
                       !((ctx->profile_mask & HD_PROFILE_FIRST_ONLY) && ctx->profile_seen[type]);
    if (timed) ctx->profile_seen[type] = true;
    if (timed && cudaEventRecord(ctx->ev_begin[slot], stream) != cudaSuccess) return HD_ERR_CUDA;
    st = cuda_status(launch_layer(km, vm, a, L.batch, ctx->group, ctx->consumer, stages,
                                  L.pdl && !timed, stream));
    if (st != HD_OK) return st;
    ++ctx->launches;
    if (timed) {
        if (cudaEventRecord(ctx->ev_end[slot], stream) != cudaSuccess) return HD_ERR_CUDA;
        ++ctx->ev_used[type];
    }
    return HD_OK;
}

// Split of a step grid: one chunk size C (a multiple of kChunkMin keys, up to
// the cache type's chunk maximum) for every layer, each layer then taking
// ceil(max_keys / C) chunks per (sequence, kv head).  C minimises an estimate
// of the grid's time in key-reads per SM, each CTA costing its keys plus a
// fixed cost for its start and combine of about 256 KiB of streaming (256
// bf16 or 512 E4M3 keys; fitted to batch-4 131k-context steps, where
// 2048-key bf16 chunks beat shorter ones): a grid that is resident at once
// (two CTAs per SM in the model, also for the E4M3 grids that hold three) ends
// with its most loaded SM, ceil(CTAs / SMs) CTAs of up to C keys; a longer grid
// takes the total over the SMs plus one CTA of tail.
int32_t plan_step_chunk(const hd_ctx *ctx, const std::vector<LayerCall> &calls, size_t rows, bool mt) {
    const int n = (int)calls.size();
    std::vector<int32_t> batch(n), max_keys(n);
    std::vector<uint8_t> one(n);
    for (int i = 0; i < n; ++i) {
        batch[i] = calls[i].batch;
        max_keys[i] = calls[i].max_keys;
        one[i] = calls[i].one_chunk ? 1 : 0;
    }
    return plan_step(ctx->cfg.num_kv_heads, ctx->num_sms, ctx->kv_type, rows, mt, n, batch.data(), max_keys.data(),
                     one.data());
}

}  // namespace

int32_t hd::plan_step(int64_t Hkv, int64_t sms, int kv_type, size_t rows, bool mt, int n, const int32_t *batch,
                      const int32_t *max_keys, const uint8_t *one_chunk) {
    const int64_t cmax = kv_type == KV_FP8 ? 2 * kChunkMax : kChunkMax;
    const int64_t fixed = (256 << 10) / (kHeadDim * kv_elem_bytes(kv_type) * 2);   // keys
    const int stages = step_stages(kv_type, rows, mt);
    int64_t longest = 1;
    for (int i = 0; i < n; ++i) longest = std::max<int64_t>(longest, max_keys[i]);
    int64_t best_c = cmax;
    double best = -1.0;
    for (int64_t C = kChunkMin; C <= cmax; C += kChunkMin) {
        int64_t ctas = 0;
        double total = 0.0;
        bool fits = true;
        for (int i = 0; i < n; ++i) {
            const int64_t Cl = one_chunk[i] ? std::max<int64_t>(C, max_keys[i]) : C;
            const int64_t ch = max_keys[i] > 0 ? (max_keys[i] + Cl - 1) / Cl : 1;
            ctas += (int64_t)batch[i] * Hkv * ch;
            total += (double)batch[i] * Hkv * (double)(ch * fixed + max_keys[i]);
            fits = fits && combine_fits(rows, ch, mt, stages);
        }
        if (!fits) continue;
        const double per_cta = (double)(std::min(C, longest) + fixed);
        const double est = ctas <= 2 * sms ? (double)((ctas + sms - 1) / sms) * per_cta : total / sms + per_cta;
        if (best < 0.0 || est <= best) {   // ties: the longer chunk
            best = est;
            best_c = C;
        }
        if (C >= longest) break;   // longer chunks change nothing
    }
    return (int32_t)best_c;
}

namespace {

// Launches the layers of one pass as step grids: layers share a grid while the
// grid has at most kStepLayers layers and their partials fit the workspace; a
// layer whose partials alone do not fit runs its own launch.  The layers are
// independent, so they go in longest first (a stable sort on their key bound):
// the long full-layer CTAs start early and the short sliding ones fill the
// grid's tail (measured 0.6-1.4 % faster steps than model order).
hd_status launch_step_calls(hd_ctx *ctx, const std::vector<LayerCall> &calls, cudaStream_t stream) {
    if (calls.empty()) return HD_OK;
    const int64_t Hkv = ctx->cfg.num_kv_heads;
    const size_t rows = (size_t)ctx->group * calls[0].tokens;
    const bool mt = calls[0].total_tokens > 1;
    const int32_t C = plan_step_chunk(ctx, calls, rows, mt);
    StepTable &t = ctx->step_table;
    int64_t part_row = 0, ctas = 0;
    std::vector<int> &order = ctx->step_order;
    order.resize(calls.size());
    for (size_t i = 0; i < order.size(); ++i) order[i] = (int)i;
    std::stable_sort(order.begin(), order.end(),
                     [&](int x, int y) { return calls[x].max_keys > calls[y].max_keys; });
    t.num_layers = 0;
    auto flush = [&]() -> hd_status {
        if (t.num_layers == 0) return HD_OK;
        const int stages = rows > (size_t)kMaxGroup ? deep_stages_for(rows)
                           : ctas <= ctx->num_sms  ? kDeepStages
                                                   : step_stages(ctx->kv_type, rows, mt);
        const size_t slot = 2 * (size_t)kProfileEvents + ctx->ev_used[2];
        const bool timed = (ctx->profile_mask & HD_PROFILE_STEP) && ctx->ev_used[2] < (size_t)kProfileEvents;
        if (timed && cudaEventRecord(ctx->ev_begin[slot], stream) != cudaSuccess) return HD_ERR_CUDA;
        hd_status st = cuda_status(launch_step(t, (int)ctas, (int)rows, mt, ctx->kv_type, ctx->consumer, stages, stream));
        if (st != HD_OK) return st;
        ++ctx->launches;
        if (timed) {
            if (cudaEventRecord(ctx->ev_end[slot], stream) != cudaSuccess) return HD_ERR_CUDA;
            ++ctx->ev_used[2];
        }
        t.num_layers = 0;
        part_row = ctas = 0;
        return HD_OK;
    };
    for (int oi : order) {
        const LayerCall &L = calls[oi];
        const int64_t Cl = L.one_chunk ? std::max<int64_t>(C, L.max_keys) : C;
        const int64_t ch = L.max_keys > 0 ? (L.max_keys + Cl - 1) / Cl : 1;
        const int64_t need = ch > 1 ? (int64_t)L.batch * Hkv * (int64_t)rows * ch : 0;
        const int64_t layer_ctas = (int64_t)L.batch * Hkv * ch;
        hd_status st = HD_OK;
        // Too large for a shared grid (its partials, its combine's shared memory at
        // this chunk count, or its CTA count): its own plan and launch, in stream order.
        if (need > ctx->part_rows || layer_ctas > INT_MAX ||
            !combine_fits(rows, ch, mt, step_stages(ctx->kv_type, rows, mt))) {
            if ((st = flush()) != HD_OK || (st = launch_layer_call(ctx, L, stream)) != HD_OK) return st;
            continue;
        }
        if (t.num_layers == kStepLayers || part_row + need > ctx->part_rows || ctas + layer_ctas > INT_MAX)
            if ((st = flush()) != HD_OK) return st;
        const CUtensorMap *km = nullptr, *vm = nullptr;
        if ((st = maps_for(ctx, L.layer, L.cache, L.batch, wide_stage_pass(ctx->kv_type, rows, ctx->consumer == CONSUMER_UMMA),
                           &km, &vm)) != HD_OK)
            return st;
        LayerLaunch &e = t.layer[t.num_layers++];
        e.kmap = *km;
        e.vmap = *vm;
        fill_layer_args(ctx, L, (int32_t)Cl, (int32_t)ch, part_row, e.a);
        t.begin[t.num_layers - 1] = (int32_t)ctas;
        part_row += need;
        ctas += layer_ctas;
    }
    return flush();
}

uint8_t *stage_row(const hd_ctx *ctx, uint8_t *base, int layer) {
    return base + (size_t)layer * ctx->cfg.max_batch * ctx->cfg.num_kv_heads * kHeadDim * kv_elem_bytes(ctx->kv_type);
}

// Host checks shared by the attention entry points and decode_step.
hd_status check_attention(const hd_ctx *ctx, int layer, int batch, const int32_t *context,
                          const hd_kv_cache &cache, const void *out, const float *lse) {
    hd_status st = check_call(ctx, layer, batch, context);
    if (st != HD_OK) return st;
    if (!out || !lse) return HD_ERR_INVALID_ARG;
    if ((st = check_cache(ctx, cache)) != HD_OK) return st;
    if (ctx->layer_types[layer] == HD_SLIDING && cache.capacity != sliding_capacity(ctx))
        return HD_ERR_CAPACITY;
    return HD_OK;
}

// Bound on every context[b] of a full-layer call (0: max_context); the last of
// `tokens` new tokens must have a table row and a cache entry.
hd_status full_hint(const hd_ctx *ctx, int32_t max_context_hint, const hd_kv_cache &cache, int *hint,
                    int tokens = 1) {
    if (max_context_hint < 0) return HD_ERR_INVALID_ARG;
    *hint = max_context_hint == 0 ? ctx->cfg.max_context - (tokens - 1) : max_context_hint;
    if (*hint < 0 || *hint + tokens - 1 > ctx->cfg.max_context) return HD_ERR_CAPACITY;
    if (*hint + tokens > cache.capacity) return HD_ERR_CAPACITY;
    return HD_OK;
}

// Whether no layer of a step call writes memory (out, lse, caches) that another
// layer of the call reads or writes, so that all layers can run in one grid.
// The verdict for the last array checked is kept (a memcmp decides reuse).
bool layers_independent(hd_ctx *ctx, int batch, int tokens, const hd_layer_io *layers) {
    const size_t n_layers = (size_t)ctx->cfg.num_layers;
    if (ctx->indep_batch == batch && ctx->indep_tokens == tokens && ctx->indep_layers.size() == n_layers &&
        std::memcmp(ctx->indep_layers.data(), layers, n_layers * sizeof(hd_layer_io)) == 0)
        return ctx->indep_ok;
    struct Range {
        uintptr_t begin, end;
        int layer;
        bool written;
    };
    std::vector<Range> r;
    r.reserve(n_layers * 11);
    auto add = [&](const void *p, size_t bytes, int layer, bool written) {
        if (p && bytes) r.push_back({(uintptr_t)p, (uintptr_t)p + bytes, layer, written});
    };
    const size_t Hq = ctx->cfg.num_q_heads, Hkv = ctx->cfg.num_kv_heads, D = kHeadDim;
    const size_t qrows = (size_t)batch * tokens * Hq, kvrows = (size_t)batch * tokens * Hkv;
    const size_t es = (size_t)kv_elem_bytes(ctx->kv_type);
    for (int i = 0; i < (int)n_layers; ++i) {
        const hd_layer_io &io = layers[i];
        add(io.q, qrows * D * 2, i, false);
        add(io.k, kvrows * D * 2, i, false);
        add(io.v, kvrows * D * 2, i, false);
        add(io.sink, Hq * sizeof(float), i, false);
        add(io.gate, qrows * sizeof(float), i, false);
        add(io.cache.k_scale, Hkv * sizeof(float), i, false);
        add(io.cache.v_scale, Hkv * sizeof(float), i, false);
        add(io.out, qrows * D * 2, i, true);
        add(io.lse, qrows * sizeof(float), i, true);
        const size_t extent = ((size_t)(batch - 1) * io.cache.seq_stride + Hkv * io.cache.capacity * D) * es;
        add(io.cache.k, extent, i, true);
        add(io.cache.v, extent, i, true);
    }
    std::sort(r.begin(), r.end(), [](const Range &x, const Range &y) { return x.begin < y.begin; });
    bool ok = true;
    for (size_t a = 0; a < r.size() && ok; ++a)
        for (size_t b = a + 1; b < r.size() && r[b].begin < r[a].end; ++b)
            if (r[a].layer != r[b].layer && (r[a].written || r[b].written)) {
                ok = false;
                break;
            }
    ctx->indep_layers.assign(layers, layers + n_layers);
    ctx->indep_batch = batch;
    ctx->indep_tokens = tokens;
    ctx->indep_ok = ok;
    return ok;
}

}  // namespace

extern "C" {

const char *hd_status_string(hd_status s) {
    switch (s) {
    case HD_OK: return "ok";
    case HD_ERR_INVALID_ARG: return "invalid argument";
    case HD_ERR_UNSUPPORTED: return "unsupported shape";
    case HD_ERR_CAPACITY: return "capacity exceeded";
    case HD_ERR_CUDA: return "CUDA error";
    case HD_ERR_STATE: return "invalid state";
    }
    return "unknown status";
}

hd_status hd_validate_config(const hd_config *cfg) {
    if (!cfg || cfg->num_layers <= 0 || !cfg->layer_types) return HD_ERR_INVALID_ARG;
    if (cfg->num_q_heads <= 0 || cfg->num_kv_heads <= 0) return HD_ERR_INVALID_ARG;
    if (cfg->num_q_heads % cfg->num_kv_heads != 0) return HD_ERR_INVALID_ARG;
    for (int i = 0; i < cfg->num_layers; ++i)
        if (cfg->layer_types[i] != HD_SLIDING && cfg->layer_types[i] != HD_FULL)
            return HD_ERR_INVALID_ARG;
    if (cfg->cache_layout != HD_LAYOUT_AUTO && cfg->cache_layout != HD_LAYOUT_RING &&
        cfg->cache_layout != HD_LAYOUT_ROLL)
        return HD_ERR_INVALID_ARG;
    if (cfg->kv_dtype != HD_KV_BF16 && cfg->kv_dtype != HD_KV_FP8_E4M3) return HD_ERR_INVALID_ARG;
    if (cfg->sliding_window < 2 || cfg->max_batch <= 0 || cfg->max_context < 0)
        return HD_ERR_INVALID_ARG;
    if (cfg->max_batch > 65535) return HD_ERR_CAPACITY;
    for (int rot : {cfg->rotary_dim_sliding, cfg->rotary_dim_full})
        if (rot < 0 || rot % 2 != 0 || rot > cfg->head_dim) return HD_ERR_INVALID_ARG;
    if (!(cfg->rope_theta_sliding > 0.0) || !(cfg->rope_theta_full > 0.0)) return HD_ERR_INVALID_ARG;
    if (cfg->head_dim != kHeadDim) return HD_ERR_UNSUPPORTED;
    const int g = cfg->num_q_heads / cfg->num_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8) return HD_ERR_UNSUPPORTED;
    return HD_OK;
}

hd_status hd_plan_split(int32_t batch, int32_t num_kv_heads, int32_t max_keys, int32_t num_sms,
                        int32_t *chunk_keys, int32_t *num_chunks) {
    if (batch <= 0 || num_kv_heads <= 0 || max_keys < 0 || num_sms <= 0 || !chunk_keys || !num_chunks)
        return HD_ERR_INVALID_ARG;
    plan_split(batch, num_kv_heads, max_keys, num_sms, INT64_MAX, chunk_keys, num_chunks);
    return HD_OK;
}

hd_status hd_plan_step_split(int32_t num_layers, const int32_t *max_keys, const uint8_t *one_chunk,
                             int32_t batch, int32_t num_kv_heads, int32_t rows, int32_t multi_token,
                             int32_t kv_dtype, int32_t num_sms, int32_t *chunk_keys) {
    if (num_layers <= 0 || !max_keys || batch <= 0 || num_kv_heads <= 0 || rows <= 0 || rows > kMaxRows ||
        (multi_token != 0 && multi_token != 1) || num_sms <= 0 || !chunk_keys ||
        (kv_dtype != HD_KV_BF16 && kv_dtype != HD_KV_FP8_E4M3))
        return HD_ERR_INVALID_ARG;
    std::vector<int32_t> b(num_layers, batch);
    std::vector<uint8_t> one(num_layers, 0);
    for (int i = 0; i < num_layers; ++i) {
        if (max_keys[i] < 0) return HD_ERR_INVALID_ARG;
        if (one_chunk) one[i] = one_chunk[i] ? 1 : 0;
    }
    *chunk_keys = plan_step(num_kv_heads, num_sms, kv_dtype == HD_KV_FP8_E4M3 ? KV_FP8 : KV_BF16, (size_t)rows,
                            multi_token != 0, num_layers, b.data(), max_keys, one.data());
    return HD_OK;
}

hd_status hybrid_decode_init(const hd_config *cfg, hd_ctx **out_ctx) {
    if (!out_ctx) return HD_ERR_INVALID_ARG;
    *out_ctx = nullptr;
    hd_status st = hd_validate_config(cfg);
    if (st != HD_OK) return st;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HD_ERR_STATE;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return HD_ERR_STATE;
    if (prop.major != 10 || prop.minor != 3) return HD_ERR_UNSUPPORTED;  // built for sm_103a only
    if (!encode_fn()) return HD_ERR_CUDA;

    hd_ctx *ctx = new (std::nothrow) hd_ctx();
    if (!ctx) return HD_ERR_CAPACITY;
    ctx->cfg = *cfg;
    ctx->layer_types.assign(cfg->layer_types, cfg->layer_types + cfg->num_layers);
    ctx->cfg.layer_types = ctx->layer_types.data();
    ctx->device = dev;
    ctx->num_sms = prop.multiProcessorCount;
    ctx->group = cfg->num_q_heads / cfg->num_kv_heads;
    ctx->sliding_layout = cfg->cache_layout == HD_LAYOUT_ROLL ? HD_LAYOUT_ROLL : HD_LAYOUT_RING;
    ctx->kv_type = cfg->kv_dtype == HD_KV_FP8_E4M3 ? KV_FP8 : KV_BF16;
    ctx->maps.resize(cfg->num_layers);
    ctx->cluster_max = layer_cluster_limit(ctx->group, ctx->kv_type);

    bool any_sliding = false, any_full = false;
    for (int t : ctx->layer_types) (t == HD_SLIDING ? any_sliding : any_full) = true;
    st = HD_OK;
    if (any_sliding)
        st = build_table(&ctx->table_sliding, cfg->rotary_dim_sliding, cfg->rope_theta_sliding,
                         cfg->max_context);
    if (st == HD_OK && any_full)
        st = build_table(&ctx->table_full, cfg->rotary_dim_full, cfg->rope_theta_full,
                         cfg->max_context);
    if (st != HD_OK) {
        free_ctx(ctx);
        return st;
    }
    const int Hkv = cfg->num_kv_heads, B = cfg->max_batch;
    int64_t slots = 0;
    if (any_full) slots = part_slot_capacity(B, cfg->max_context + 1, ctx->num_sms);
    if (any_sliding) {
        const int64_t s = part_slot_capacity(B, cfg->sliding_window, ctx->num_sms);
        if (s > slots) slots = s;
    }
    ctx->part_slots = slots;
    // Partial rows: a single-layer call holds up to kMaxRows rows per kv head
    // (query heads, or heads x tokens) for each of its slots.  A step grid holds
    // those of all its multi-chunk layers at once: at full batch and the longest
    // chunk, or at most two CTAs per SM for short steps; up to 2^20 rows (1 GiB),
    // beyond which a step runs as several grids.
    int64_t fused = 2LL * ctx->num_sms * kMaxRows;
    const int64_t cmax = ctx->kv_type == KV_FP8 ? 2 * kChunkMax : kChunkMax;
    for (int t : ctx->layer_types) {
        const int64_t keys = t == HD_FULL ? (int64_t)cfg->max_context + kMaxTokens : cfg->sliding_window;
        const int64_t ch = (keys + cmax - 1) / cmax;
        if (ch > 1) fused += (int64_t)B * Hkv * kMaxRows * ch;
    }
    ctx->part_rows = std::max<int64_t>(slots * Hkv * kMaxRows, std::min<int64_t>(fused, 1LL << 20));
    const size_t counters = (size_t)cfg->num_layers * B * Hkv * sizeof(int32_t);
    bool ok = cudaMalloc(&ctx->part_o, (size_t)ctx->part_rows * kHeadDim * sizeof(float)) == cudaSuccess &&
              cudaMalloc(&ctx->part_ml, (size_t)ctx->part_rows * sizeof(float2)) == cudaSuccess &&
              cudaMalloc(&ctx->counters, counters) == cudaSuccess &&
              cudaMemset(ctx->counters, 0, counters) == cudaSuccess &&
              cudaMalloc(&ctx->err, sizeof(int32_t)) == cudaSuccess &&
              cudaMemset(ctx->err, 0, sizeof(int32_t)) == cudaSuccess;
    const size_t stage = (size_t)cfg->num_layers * B * Hkv * kHeadDim * kv_elem_bytes(ctx->kv_type);
    ok = ok && cudaMalloc(&ctx->stage_k, stage) == cudaSuccess && cudaMalloc(&ctx->stage_v, stage) == cudaSuccess;
    // The tables, zeroed counters and error word are complete before any call, on
    // whatever stream the caller uses (a non-blocking stream is not ordered after
    // the legacy-stream copies and memsets above).
    ok = ok && cudaDeviceSynchronize() == cudaSuccess;
    if (!ok) {
        free_ctx(ctx);
        return HD_ERR_CUDA;
    }
    *out_ctx = ctx;
    return HD_OK;
}

hd_status hybrid_decode_destroy(hd_ctx *ctx) {
    if (!ctx) return HD_ERR_INVALID_ARG;
    cudaDeviceSynchronize();
    free_ctx(ctx);
    return HD_OK;
}

hd_status rope_append_kv(hd_ctx *ctx, int32_t layer, int32_t batch, const int32_t *context,
                         const void *q, const void *k, const void *v, float *q_rot,
                         hd_kv_cache cache, void *stream) {
    hd_status st = check_call(ctx, layer, batch, context);
    if (st != HD_OK || (st = check_device(ctx)) != HD_OK) return st;
    if (!q || !k || !v || !q_rot || !aligned16(q_rot)) return HD_ERR_INVALID_ARG;
    if ((st = check_cache(ctx, cache)) != HD_OK) return st;
    const bool sliding = ctx->layer_types[layer] == HD_SLIDING;
    if (sliding && cache.capacity != sliding_capacity(ctx)) return HD_ERR_CAPACITY;
    const DeviceTable &tab = sliding ? ctx->table_sliding : ctx->table_full;
    const int key_set = !sliding ? KEYS_FULL_CACHED
                                 : (ctx->sliding_layout == HD_LAYOUT_ROLL ? KEYS_ROLL : KEYS_RING);
    RopeArgs a{};
    a.context = context;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k = static_cast<const __nv_bfloat16 *>(k);
    a.v = static_cast<const __nv_bfloat16 *>(v);
    a.q_rot = q_rot;
    a.table = tab.data;
    a.err = ctx->err;
    a.num_q_heads = ctx->cfg.num_q_heads;
    a.num_kv_heads = ctx->cfg.num_kv_heads;
    a.rotary_dim = tab.rotary_dim;
    a.key_set = key_set;
    a.window = ctx->cfg.sliding_window;
    a.max_context = ctx->cfg.max_context;
    a.kv_type = ctx->kv_type;
    a.k_scale = cache.k_scale;
    a.v_scale = cache.v_scale;
    if (key_set == KEYS_RING) {
        a.dst_k = stage_row(ctx, ctx->stage_k, layer);
        a.dst_v = stage_row(ctx, ctx->stage_v, layer);
        a.seq_stride = (int64_t)ctx->cfg.num_kv_heads * kHeadDim;
        a.capacity = 1;
    } else {
        a.dst_k = cache.k;
        a.dst_v = cache.v;
        a.seq_stride = cache.seq_stride;
        a.capacity = cache.capacity;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = cuda_status(launch_rope_append(a, batch, s));
    if (st != HD_OK) return st;
    ++ctx->launches;
    if (key_set == KEYS_ROLL) {
        st = cuda_status(launch_roll_window(a, batch, s));
        if (st == HD_OK) ++ctx->launches;
    }
    return st;
}

hd_status decode_attn_sliding(hd_ctx *ctx, int32_t layer, int32_t batch, const int32_t *context,
                              const float *q_rot, hd_kv_cache cache, const float *sink, const float *gate,
                              void *out, float *lse, void *stream) {
    hd_status st = check_attention(ctx, layer, batch, context, cache, out, lse);
    if (st != HD_OK || (st = check_device(ctx)) != HD_OK) return st;
    if (ctx->layer_types[layer] != HD_SLIDING) return HD_ERR_STATE;
    if (!q_rot || !aligned16(q_rot)) return HD_ERR_INVALID_ARG;
    const bool roll = ctx->sliding_layout == HD_LAYOUT_ROLL;
    LayerCall L{};
    L.layer = layer;
    L.batch = batch;
    L.context = context;
    L.max_keys = roll ? ctx->cfg.sliding_window : cache.capacity;
    L.key_set = roll ? KEYS_ROLL : KEYS_RING;
    L.new_kind = roll ? NEW_NONE : NEW_STAGED;
    L.commit = roll ? COMMIT_NONE : COMMIT_RING;
    L.q_rot = q_rot;
    L.new_k = stage_row(ctx, ctx->stage_k, layer);
    L.new_v = stage_row(ctx, ctx->stage_v, layer);
    L.cache = cache;
    L.sink = sink;
    L.gate = gate;
    L.out = out;
    L.lse = lse;
    ctx->profile_seen[0] = ctx->profile_seen[1] = false;   // each standalone call is its own step
    return launch_layer_call(ctx, L, static_cast<cudaStream_t>(stream));
}

hd_status decode_attn_full(hd_ctx *ctx, int32_t layer, int32_t batch, const int32_t *context,
                           int32_t max_context_hint, const float *q_rot, hd_kv_cache cache,
                           const float *sink, const float *gate, void *out, float *lse, void *stream) {
    hd_status st = check_attention(ctx, layer, batch, context, cache, out, lse);
    if (st != HD_OK || (st = check_device(ctx)) != HD_OK) return st;
    if (ctx->layer_types[layer] != HD_FULL) return HD_ERR_STATE;
    if (!q_rot || !aligned16(q_rot)) return HD_ERR_INVALID_ARG;
    int hint = 0;
    if ((st = full_hint(ctx, max_context_hint, cache, &hint)) != HD_OK) return st;
    LayerCall L{};
    L.layer = layer;
    L.batch = batch;
    L.context = context;
    L.max_keys = hint + 1;
    L.key_set = KEYS_FULL_CACHED;
    L.new_kind = NEW_NONE;
    L.commit = COMMIT_NONE;
    L.q_rot = q_rot;
    L.cache = cache;
    L.sink = sink;
    L.gate = gate;
    L.out = out;
    L.lse = lse;
    ctx->profile_seen[0] = ctx->profile_seen[1] = false;   // each standalone call is its own step
    return launch_layer_call(ctx, L, static_cast<cudaStream_t>(stream));
}

// q is rotated in the CTA prologue, the new key is rotated, scored and stored
// by the combine (roll layouts shift first).
hd_status decode_step(hd_ctx *ctx, int32_t batch, const int32_t *context, int32_t max_context_hint,
                      const hd_layer_io *layers, void *stream) {
    return decode_step_tokens(ctx, batch, 1, context, max_context_hint, layers, stream);
}

// T tokens per sequence: each layer runs in passes of up to 32 (bf16 caches: the
// tcgen05 pass) or 16 rows / group tokens (a power of two, at most kMaxTokens),
// the tokens of a pass being extra query rows that share one stream of the
// cache; passes of more than kMaxGroup rows run one CTA per SM on a deep ring.  A pass commits its entries, so the next pass
// (launched in full stream order) sees them as cached keys at context + token0.
hd_status decode_step_tokens(hd_ctx *ctx, int32_t batch, int32_t num_tokens, const int32_t *context,
                             int32_t max_context_hint, const hd_layer_io *layers, void *stream) {
    if (!ctx || !layers || num_tokens < 1 || num_tokens > kMaxTokens) return HD_ERR_INVALID_ARG;
    if (check_device(ctx) != HD_OK) return HD_ERR_STATE;
    if (num_tokens > 1 && !tensor_consumer(ctx->consumer)) return HD_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ctx->profile_seen[0] = ctx->profile_seen[1] = false;
    // Every layer is checked before anything is launched.
    for (int i = 0; i < ctx->cfg.num_layers; ++i) {
        const hd_layer_io &io = layers[i];
        hd_status st = check_attention(ctx, i, batch, context, io.cache, io.out, io.lse);
        if (st != HD_OK) return st;
        if (!io.q || !io.k || !io.v || !aligned16(io.q) || !aligned16(io.k) || !aligned16(io.v))
            return HD_ERR_INVALID_ARG;
    }
    // Independent layers (the call's contract) may share one grid, or overlap as
    // one kernel per layer; layers that alias run one kernel per layer in full order.
    const bool indep = layers_independent(ctx, batch, num_tokens, layers);
    const bool fused = ctx->fuse_step && tensor_consumer(ctx->consumer) && indep;
    std::vector<LayerCall> &calls = ctx->step_calls;
    calls.assign(ctx->cfg.num_layers, LayerCall{});
    for (int i = 0; i < ctx->cfg.num_layers; ++i) {
        const hd_layer_io &io = layers[i];
        hd_status st = HD_OK;
        const bool sliding = ctx->layer_types[i] == HD_SLIDING;
        const bool roll = sliding && ctx->sliding_layout == HD_LAYOUT_ROLL;
        LayerCall &L = calls[i];
        L.layer = i;
        L.batch = batch;
        L.context = context;
        L.q_bf16 = io.q;
        L.new_k = io.k;
        L.new_v = io.v;
        L.cache = io.cache;
        L.sink = io.sink;
        L.gate = io.gate;
        L.out = io.out;
        L.lse = io.lse;
        L.total_tokens = num_tokens;
        if (!sliding) {
            int hint = 0;
            if ((st = full_hint(ctx, max_context_hint, io.cache, &hint, num_tokens)) != HD_OK) return st;
            L.max_keys = hint + num_tokens - 1;
            L.key_set = KEYS_FULL_PREV;
            L.new_kind = NEW_ROTATE;
            L.commit = COMMIT_APPEND;
        } else if (!roll) {
            L.max_keys = io.cache.capacity;
            L.key_set = KEYS_RING;
            L.new_kind = NEW_ROTATE;
            L.commit = COMMIT_RING;
        } else {   // the kernel reads the window, then shifts it and stores the new entries
            L.max_keys = ctx->cfg.sliding_window - 1;
            L.key_set = KEYS_ROLL_SHIFT;
            L.new_kind = NEW_ROTATE;
            L.commit = COMMIT_ROLL;
            L.one_chunk = true;
        }
    }
    // rows per pass: up to 32 with bf16 caches (the tcgen05 pass), else 16
    const int rows_cap = ctx->kv_type == KV_BF16 ? kMaxRows : kMaxRowsMma;
    const int tmax = std::min(kMaxTokens, rows_cap / ctx->group);
    if (fused) {
        // Step grids, pass by pass: a pass commits its entries, and the next pass's
        // grid starts after it in full stream order.
        for (int t0 = 0; t0 < num_tokens;) {
            int tp = 1;
            while (2 * tp <= tmax && 2 * tp <= num_tokens - t0) tp *= 2;
            for (LayerCall &L : calls) {
                L.tokens = tp;
                L.token0 = t0;
                L.pdl = false;
            }
            hd_status st = launch_step_calls(ctx, calls, s);
            if (st != HD_OK) return st;
            t0 += tp;
        }
        return HD_OK;
    }
    // One kernel per layer (and pass); a layer's first pass may start streaming
    // while the previous layer drains.
    for (LayerCall &L : calls) {
        for (int t0 = 0; t0 < num_tokens;) {
            int tp = 1;
            while (2 * tp <= tmax && 2 * tp <= num_tokens - t0) tp *= 2;
            L.tokens = tp;
            L.token0 = t0;
            // Every layer after the first is a programmatic dependent of the previous
            // kernel: independent layers with overlap on read and stream before it
            // completes; otherwise (full stream order) they wait before their first read.
            // (A later pass reads what the previous pass wrote.)
            L.pdl = L.layer > 0 && t0 == 0;
            L.early = indep && ctx->layer_overlap;
            hd_status st = launch_layer_call(ctx, L, s);
            if (st != HD_OK) return st;
            t0 += tp;
        }
    }
    return HD_OK;
}

hd_status hybrid_decode_set_step_fusion(hd_ctx *ctx, int32_t enable) {
    if (!ctx || (enable != 0 && enable != 1)) return HD_ERR_INVALID_ARG;
    ctx->fuse_step = enable != 0;
    return HD_OK;
}

hd_status hybrid_decode_set_cluster_combine(hd_ctx *ctx, int32_t enable) {
    if (!ctx || (enable != 0 && enable != 1)) return HD_ERR_INVALID_ARG;
    ctx->cluster_combine = enable != 0;
    return HD_OK;
}

hd_status hybrid_decode_set_layer_overlap(hd_ctx *ctx, int32_t enable) {
    if (!ctx || (enable != 0 && enable != 1)) return HD_ERR_INVALID_ARG;
    ctx->layer_overlap = enable != 0;
    return HD_OK;
}

hd_status hybrid_decode_inject_lost_copy(hd_ctx *ctx, int32_t stage) {
    if (!ctx || stage < -1) return HD_ERR_INVALID_ARG;
    ctx->drop_stage = stage;
    return HD_OK;
}

hd_status hybrid_decode_set_consumer(hd_ctx *ctx, int32_t consumer) {
    if (!ctx) return HD_ERR_INVALID_ARG;
    switch (consumer) {
    case HD_CONSUMER_CUDA_CORE: ctx->consumer = CONSUMER_FMA; break;
    case HD_CONSUMER_TENSOR_CORE: ctx->consumer = CONSUMER_MMA; break;
    case HD_CONSUMER_TENSOR_MEMORY: ctx->consumer = CONSUMER_UMMA; break;
    default: return HD_ERR_INVALID_ARG;
    }
    return HD_OK;
}

hd_status hybrid_decode_device_errors(hd_ctx *ctx, int32_t *flags, void *stream) {
    if (!ctx || !flags) return HD_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t host = 0;
    if (cudaMemcpyAsync(&host, ctx->err, sizeof host, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(ctx->err, 0, sizeof host, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return HD_ERR_CUDA;
    *flags = host;
    return HD_OK;
}

hd_status hybrid_decode_launch_count(hd_ctx *ctx, int64_t *launches) {
    if (!ctx || !launches) return HD_ERR_INVALID_ARG;
    *launches = ctx->launches;
    return HD_OK;
}

hd_status hybrid_decode_set_profiling(hd_ctx *ctx, int32_t enable) {
    if (!ctx || enable < 0 || enable > (HD_PROFILE_SLIDING | HD_PROFILE_FULL | HD_PROFILE_FIRST_ONLY | HD_PROFILE_STEP))
        return HD_ERR_INVALID_ARG;
    if (enable && ctx->ev_begin.empty()) {
        ctx->ev_begin.resize(3 * kProfileEvents);
        ctx->ev_end.resize(3 * kProfileEvents);
        for (int i = 0; i < 3 * kProfileEvents; ++i)
            if (cudaEventCreate(&ctx->ev_begin[i]) != cudaSuccess ||
                cudaEventCreate(&ctx->ev_end[i]) != cudaSuccess)
                return HD_ERR_CUDA;
    }
    ctx->profile_mask = enable;
    ctx->ev_used[0] = ctx->ev_used[1] = ctx->ev_used[2] = 0;
    return HD_OK;
}

hd_status hybrid_decode_profile(hd_ctx *ctx, int32_t layer_type, double *total_ms, int64_t *launches) {
    if (!ctx || !total_ms || !launches) return HD_ERR_INVALID_ARG;
    if (layer_type != HD_SLIDING && layer_type != HD_FULL && layer_type != HD_PROFILE_KIND_STEP)
        return HD_ERR_INVALID_ARG;
    double sum = 0.0;
    const size_t n = ctx->ev_used[layer_type];
    for (size_t i = 0; i < n; ++i) {
        const size_t slot = (size_t)layer_type * kProfileEvents + i;
        if (cudaEventSynchronize(ctx->ev_end[slot]) != cudaSuccess) return HD_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, ctx->ev_begin[slot], ctx->ev_end[slot]) != cudaSuccess)
            return HD_ERR_CUDA;
        sum += ms;
    }
    *total_ms = sum;
    *launches = (int64_t)n;
    ctx->ev_used[layer_type] = 0;
    return HD_OK;
}

}  // extern "C"
