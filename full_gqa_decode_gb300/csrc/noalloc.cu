// decode_attn_full_static_scratch: full-layer decode attention that allocates
// nothing, for callers that cannot call cudaMalloc.
//
// Who needs it: host programs that must not allocate device memory once they
// are running -- a plugin living inside a runtime that owns and pre-plans
// every device allocation, or a serving loop on a latency budget, where
// cudaMalloc/cudaFree may synchronise the device or fail under a fixed memory
// plan.  Those callers cannot create an hd_ctx (hybrid_decode_init allocates
// its workspace), so this entry point needs no context: the caller passes the
// inputs and outputs, and the split-K scratch (chunk partials, chunk tickets,
// the device error word) lives in one file-scope device array below.
//
// That array is part of the loaded library: every GPU on which the library is
// used holds kScratchBytes of it until the process exits.  All calls share it
// and it keeps the last call's contents, so two calls that overlap on the GPU
// (different streams, or different host threads without ordering) race on it
// and give wrong results; order such calls on one stream.
//
// Setup: the first call in a CUDA context (per device, with that device
// current) looks up the array's device address with cudaGetSymbolAddress and
// caches it together with the context's id (in host code the array's name is
// only a host-side stand-in, not a device address).  A context that was torn
// down and made again (cudaDeviceReset) has a new id, so its first call looks
// the address up again.  Make the first call before any stream capture.
#include <cudaTypedefs.h>

#include <mutex>

#include "hd_internal.h"

namespace {

constexpr size_t kScratchBytes = HD_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Chunk partials (o, then (m, l)), then the per-(sequence, kv head) tickets and
// the device error word.  Zero-initialised at load; the tickets and the error
// word are cleared again before every launch.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct ScratchAddress {
    unsigned long long context_id = 0;
    void *ptr = nullptr;
};
std::mutex g_mutex;
ScratchAddress g_scratch_addr[kMaxDevices];

template <class F>
F driver_entry(const char *name, int version) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<F>(p);
    return nullptr;
}

// Id of the current CUDA context (0 when none is current yet or it cannot be read).
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        get_current = driver_entry<PFN_cuCtxGetCurrent_v4000>("cuCtxGetCurrent", 4000);
        get_id = driver_entry<PFN_cuCtxGetId_v12000>("cuCtxGetId", 12000);
    });
    if (!get_current || !get_id) return 0;
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (get_current(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

hd_status scratch_for_current_device(unsigned char **ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HD_ERR_STATE;
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(g_mutex);
    ScratchAddress &e = g_scratch_addr[dev];
    if (!e.ptr || id == 0 || e.context_id != id) {
        // The lookup binds the device's primary context if none is current yet.
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) {
            e = ScratchAddress{};
            return HD_ERR_CUDA;
        }
        e.ptr = p;
        e.context_id = current_context_id();
    }
    *ptr = static_cast<unsigned char *>(e.ptr);
    return HD_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] { fn = driver_entry<PFN_cuTensorMapEncodeTiled_v12000>("cuTensorMapEncodeTiled", 12000); });
    return fn;
}

// The same 4-D view and swizzled box the layer kernel's consumers index by.
bool encode(CUtensorMap *map, const void *base, const hd_kv_cache &c, int num_kv_heads, int batch) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)hd::kHeadDim, (cuuint64_t)c.capacity, (cuuint64_t)num_kv_heads,
                                (cuuint64_t)batch};
    const cuuint64_t strides[3] = {(cuuint64_t)hd::kHeadDim * 2, (cuuint64_t)c.capacity * hd::kHeadDim * 2,
                                   (cuuint64_t)c.seq_stride * 2};
    const cuuint32_t box[4] = {(cuuint32_t)hd::kBoxCols, (cuuint32_t)hd::kStageKeys, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Scratch layout of one call: partial outputs, then (m, l) pairs, then the
// tickets and the error word.
struct ScratchPlan {
    int32_t chunk_keys = 0, num_chunks = 0, stages = hd::kStages;
    size_t o_bytes = 0, ml_bytes = 0, ctr_bytes = 0, total = 0;
};

hd_status plan_scratch(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t max_context,
                       int32_t num_sms, ScratchPlan *p) {
    if (batch <= 0 || batch > 65535 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_q_heads % num_kv_heads != 0 || max_context < 0 || max_context == INT32_MAX || num_sms <= 0)
        return HD_ERR_INVALID_ARG;
    const int group = num_q_heads / num_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8) return HD_ERR_UNSUPPORTED;
    // Chunks no larger in number than the array can hold at the largest chunk size.
    const int64_t per_slot = (int64_t)num_q_heads * (hd::kHeadDim * sizeof(float) + sizeof(float2));
    hd::plan_split(batch, num_kv_heads, (int64_t)max_context + 1, num_sms, (int64_t)(kScratchBytes / 2) / per_slot,
                   &p->chunk_keys, &p->num_chunks, &p->stages);
    const size_t slots = (size_t)batch * num_q_heads * p->num_chunks;
    p->o_bytes = slots * hd::kHeadDim * sizeof(float);
    p->ml_bytes = slots * sizeof(float2);
    p->ctr_bytes = (size_t)batch * num_kv_heads * sizeof(int32_t);
    p->total = p->o_bytes + p->ml_bytes + p->ctr_bytes + sizeof(int32_t);
    if (p->total > kScratchBytes) return HD_ERR_CAPACITY;
    if (!hd::combine_fits((size_t)group, p->num_chunks, false, p->stages)) return HD_ERR_CAPACITY;
    return HD_OK;
}

}  // namespace

extern "C" hd_status decode_attn_full_static_scratch_plan(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                                          int32_t max_context, int32_t num_sms,
                                                          int64_t *scratch_bytes, int32_t *chunk_keys,
                                                          int32_t *num_chunks) {
    ScratchPlan p;
    const hd_status st = plan_scratch(batch, num_q_heads, num_kv_heads, max_context, num_sms, &p);
    if (st == HD_OK || st == HD_ERR_CAPACITY) {
        if (scratch_bytes) *scratch_bytes = (int64_t)p.total;
        if (chunk_keys) *chunk_keys = p.chunk_keys;
        if (num_chunks) *num_chunks = p.num_chunks;
    }
    return st;
}

extern "C" hd_status decode_attn_full_static_scratch(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                                     const int32_t *context, int32_t max_context,
                                                     const float *q_rot, hd_kv_cache cache,
                                                     const float *sink, void *out, float *lse,
                                                     void *stream) {
    // Arguments (host checks, before anything touches the device).
    if (!context || !q_rot || !out || !lse || !aligned16(q_rot)) return HD_ERR_INVALID_ARG;
    if (!cache.k || !cache.v || !aligned16(cache.k) || !aligned16(cache.v) || cache.capacity <= 0 ||
        cache.seq_stride % 8 != 0 || num_kv_heads <= 0 ||
        cache.seq_stride < (int64_t)num_kv_heads * cache.capacity * hd::kHeadDim)
        return HD_ERR_INVALID_ARG;
    if (cache.k_scale || cache.v_scale) return HD_ERR_UNSUPPORTED;   // bf16 caches only
    if (max_context < 0) return HD_ERR_INVALID_ARG;
    if ((int64_t)max_context + 1 > cache.capacity) return HD_ERR_CAPACITY;

    int device = 0, num_sms = 0;
    if (cudaGetDevice(&device) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return HD_ERR_STATE;
    // The split plan and the size limit: calls needing more than the array are refused.
    ScratchPlan plan;
    hd_status st = plan_scratch(batch, num_q_heads, num_kv_heads, max_context, num_sms, &plan);
    if (st != HD_OK) return st;

    unsigned char *scratch = nullptr;
    if ((st = scratch_for_current_device(&scratch)) != HD_OK) return st;
    CUtensorMap kmap, vmap;
    if (!encode(&kmap, cache.k, cache, num_kv_heads, batch) || !encode(&vmap, cache.v, cache, num_kv_heads, batch))
        return HD_ERR_CUDA;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t *counters = reinterpret_cast<int32_t *>(scratch + plan.o_bytes + plan.ml_bytes);
    if (cudaMemsetAsync(counters, 0, plan.ctr_bytes + sizeof(int32_t), s) != cudaSuccess) return HD_ERR_CUDA;

    hd::LayerArgs a{};
    a.context = context;
    a.q_rot = q_rot;
    a.new_kind = hd::NEW_NONE;
    a.commit = hd::COMMIT_NONE;
    a.key_set = hd::KEYS_FULL_CACHED;
    a.cache_k = cache.k;
    a.cache_v = cache.v;
    a.kv_type = hd::KV_BF16;
    a.seq_stride = cache.seq_stride;
    a.capacity = cache.capacity;
    a.sink = sink;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.lse = lse;
    a.part_o = reinterpret_cast<float *>(scratch);
    a.part_ml = reinterpret_cast<float2 *>(scratch + plan.o_bytes);
    a.counters = counters;
    a.err = counters + (size_t)batch * num_kv_heads;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.chunk_keys = plan.chunk_keys;
    a.max_chunks = plan.num_chunks;
    a.window = 0;
    a.max_context = max_context;
    a.drop_stage = -1;
    a.tokens = a.total_tokens = 1;
    return hd::launch_layer(&kmap, &vmap, a, batch, num_q_heads / num_kv_heads, hd::CONSUMER_MMA, plan.stages, false,
                            s) == cudaSuccess
               ? HD_OK
               : HD_ERR_CUDA;
}
