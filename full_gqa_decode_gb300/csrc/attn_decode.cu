// Single-layer launches of the attention kernel (attn_kernel.cuh) for bf16
// caches, and the host dispatch of layer and step launches.
#include "attn_kernel.cuh"

namespace hd {

// `stages` in bf16 stages: the ring's bytes; an E4M3 ring has twice as many
// (half-size) stages and so twice the mbarriers.
size_t layer_smem_bytes(int group, int stages) {
    return 1024 + (size_t)stages * kStageBytes + ((size_t)group * kHeadDim + 4 * kHeadDim + 32) * sizeof(float) +
           2 * (size_t)(2 * stages) * sizeof(uint64_t) + 16 + 16 * sizeof(unsigned) + 2 * kHeadDim +
           kMaxRows * sizeof(int);
}

int layer_cluster_limit(int group, int kv) {
    if (kv == KV_FP8) return layer_cluster_limit_fp8(group);
    switch (group) {
    case 1: return cluster_limit_g<1, KV_BF16>();
    case 2: return cluster_limit_g<2, KV_BF16>();
    case 4: return cluster_limit_g<4, KV_BF16>();
    case 8: return cluster_limit_g<8, KV_BF16>();
    default: return 0;
    }
}

cudaError_t launch_layer_bf16(const LaunchTable<1> &t, dim3 grid, int rows, bool mt, int consumer, int stages,
                              bool pdl, cudaStream_t s) {
    return launch_kv<KV_BF16, 1>(t, grid, rows, mt, consumer, stages, pdl, s);
}

cudaError_t launch_layer(const CUtensorMap *km, const CUtensorMap *vm, const LayerArgs &a, int batch,
                         int group, int consumer, int stages, bool pdl, cudaStream_t s) {
    LaunchTable<1> t;
    t.layer[0].kmap = *km;
    t.layer[0].vmap = *vm;
    t.layer[0].a = a;
    t.begin[0] = 0;
    t.num_layers = 1;
    const dim3 grid(a.max_chunks, a.num_kv_heads, batch);
    const bool mt = a.total_tokens > 1;
    const int rows = group * (mt ? a.tokens : 1);
    return a.kv_type == KV_FP8 ? launch_layer_fp8(t, grid, rows, mt, consumer, stages, pdl, s)
                               : launch_layer_bf16(t, grid, rows, mt, consumer, stages, pdl, s);
}

cudaError_t launch_step(const StepTable &t, int num_ctas, int rows, bool mt, int kv, int consumer, int stages,
                        cudaStream_t s) {
    if (t.num_layers < 1 || t.num_layers > kStepLayers || num_ctas < 1) return cudaErrorInvalidValue;
    const dim3 grid(num_ctas);
    return kv == KV_FP8 ? launch_step_fp8(t, grid, rows, mt, stages, s)
                        : launch_step_bf16(t, grid, rows, mt, consumer, stages, s);
}

}  // namespace hd
