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
// Setup: the first call on a device, with that device current, looks up the
// array's device address with cudaGetSymbolAddress and caches it for that
// device (in host code the array's name is only a host-side stand-in, not a
// device address).  Make that first call before any stream capture.
#include <cudaTypedefs.h>

#include <mutex>

#include "hd_internal.h"

namespace {

constexpr size_t kScratchBytes = 64ull << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

// Chunk partials (o, then (m, l)), then the per-(sequence, kv head) tickets and
// the device error word.  Zero-initialised at load; the tickets and the error
// word are cleared again before every launch.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

hd_status scratch_for_current_device(unsigned char **ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HD_ERR_STATE;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return HD_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *ptr = static_cast<unsigned char *>(g_scratch_ptr[dev]);
    return HD_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
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

}  // namespace

extern "C" hd_status decode_attn_full_static_scratch(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                                     const int32_t *context, int32_t max_context,
                                                     const float *q_rot, hd_kv_cache cache,
                                                     const float *sink, void *out, float *lse,
                                                     void *stream) {
    // Arguments (host checks, before anything touches the device).
    if (batch <= 0 || batch > 65535 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_q_heads % num_kv_heads != 0)
        return HD_ERR_INVALID_ARG;
    const int group = num_q_heads / num_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8) return HD_ERR_UNSUPPORTED;
    if (!context || !q_rot || !out || !lse || !aligned16(q_rot)) return HD_ERR_INVALID_ARG;
    if (!cache.k || !cache.v || !aligned16(cache.k) || !aligned16(cache.v) || cache.capacity <= 0 ||
        cache.seq_stride % 8 != 0 || cache.seq_stride < (int64_t)num_kv_heads * cache.capacity * hd::kHeadDim)
        return HD_ERR_INVALID_ARG;
    if (cache.k_scale || cache.v_scale) return HD_ERR_UNSUPPORTED;   // bf16 caches only
    if (max_context < 0) return HD_ERR_INVALID_ARG;
    if ((int64_t)max_context + 1 > cache.capacity) return HD_ERR_CAPACITY;

    int device = 0, num_sms = 0;
    if (cudaGetDevice(&device) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return HD_ERR_STATE;
    int32_t chunk_keys = 0, num_chunks = 0;
    hd_status st = HD_OK;
    // Chunks no larger in number than the array can hold at the largest chunk size.
    const int64_t per_slot = (int64_t)num_q_heads * (hd::kHeadDim * sizeof(float) + sizeof(float2));
    int32_t stages = hd::kStages;
    hd::plan_split(batch, num_kv_heads, max_context + 1, num_sms, (int64_t)(kScratchBytes / 2) / per_slot,
                   &chunk_keys, &num_chunks, &stages);

    // Scratch layout and the size limit: calls needing more than the array are refused.
    const size_t slots = (size_t)batch * num_q_heads * num_chunks;
    const size_t o_bytes = slots * hd::kHeadDim * sizeof(float);
    const size_t ml_bytes = slots * sizeof(float2);
    const size_t ctr_bytes = (size_t)batch * num_kv_heads * sizeof(int32_t);
    const size_t need = o_bytes + ml_bytes + ctr_bytes + sizeof(int32_t);
    if (need > kScratchBytes) return HD_ERR_CAPACITY;
    if (((size_t)group * num_chunks + 3) * sizeof(float) + (size_t)group * 64 * 16 >
        (size_t)hd::kStages * hd::kStageBytes)
        return HD_ERR_CAPACITY;

    unsigned char *scratch = nullptr;
    if ((st = scratch_for_current_device(&scratch)) != HD_OK) return st;
    CUtensorMap kmap, vmap;
    if (!encode(&kmap, cache.k, cache, num_kv_heads, batch) || !encode(&vmap, cache.v, cache, num_kv_heads, batch))
        return HD_ERR_CUDA;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t *counters = reinterpret_cast<int32_t *>(scratch + o_bytes + ml_bytes);
    if (cudaMemsetAsync(counters, 0, ctr_bytes + sizeof(int32_t), s) != cudaSuccess) return HD_ERR_CUDA;

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
    a.part_ml = reinterpret_cast<float2 *>(scratch + o_bytes);
    a.counters = counters;
    a.err = counters + (size_t)batch * num_kv_heads;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.chunk_keys = chunk_keys;
    a.max_chunks = num_chunks;
    a.window = 0;
    a.max_context = max_context;
    a.drop_stage = -1;
    return hd::launch_layer(&kmap, &vmap, a, batch, group, hd::CONSUMER_MMA, stages, false, s) == cudaSuccess
               ? HD_OK
               : HD_ERR_CUDA;
}
