/*
 * hybrid_decode.h -- C ABI of the GB300 (sm_103a) decode-attention library for
 * a hybrid sliding-window / full-attention GQA model.
 *
 * The operation is one autoregressive decode step of attention with the KV
 * cache passed in and out as explicit caller-owned tensors, as stated by
 * vllm_omni/edge/spark_export.py (module docstring; `SparkDecodeStep`,
 * `_Layer.forward`).  Per layer and sequence b, with c = context[b] previous
 * tokens (the new token sits at position c):
 *   - rotate q and the new k with Neox-style partial RoPE (`_rope`, `_angles`):
 *     the first rotary_dim dims as half-pairs, the rest passing through;
 *     sliding layers use their own rotary_dim/theta, full layers theirs;
 *   - score  s_j = q_rot . K_j / sqrt(head_dim)  over the layer's key set and
 *     take one softmax (`_Layer.forward`, ring and roll branches).  Query head
 *     h reads kv head h / (num_q_heads / num_kv_heads) (GQA fold);
 *   - key set: full layers score positions 0..c; sliding layers the window
 *     max(0, c-window+1)..c, the window counting the current token
 *     (`SparkStepConfig.cache_len`);
 *   - lse = log(sum_j exp(s_j)) (natural log, without the sink); with a
 *     per-head fp32 sink the output is multiplied by
 *     exp(lse) / (exp(lse) + exp(sink[h]))   (flashmla_sparse.py,
 *     `HYV4FlashMLASparseImpl` docstring); a sink of -inf is no sink;
 *   - optional output gate: with per-step gate logits g[b][h] the output is
 *     then multiplied by sigmoid(g) = 1/(1+exp(-g)) (spark_export.py
 *     `_Layer.forward`, the sigmoid of the gate projection times the
 *     attention output); lse is not gated.  The logits come from a
 *     projection outside this library and are passed in;
 *   - cache update: full layers append at index c; sliding ring layouts write
 *     slot c mod (window-1), after the cached entries have been scored; the
 *     sliding roll layout shifts its window by one once full and appends
 *     (`cache_layout` docstring; ring and roll branches).
 *
 * Numeric contract: bf16 q/k/v/caches/out (or E4M3 caches with per-kv-head
 * fp32 scales, hd_config.kv_dtype), fp32 accumulation, fp32 lse.  RoPE tables
 * hold fp32 cos/sin evaluated in fp64 at init.  The written key is
 * bf16_rne(k1*c - k2*s) / bf16_rne(k2*c + k1*s) computed in fp64 from the fp32
 * table values, so it is reproducible bit for bit; V is stored bit for bit.
 * An E4M3 entry is e4m3_rne(x / scale) of that fp64 value (of the bf16 v for
 * V), with the quotient rounded once, so it is reproducible bit for bit too.
 *
 * Memory and ownership: every tensor argument is a DEVICE pointer owned by the
 * caller (PyTorch allocates them); the library owns only the hd_ctx and the
 * device workspace it allocates in hybrid_decode_init (RoPE tables, split-K
 * partials, the ring staging rows).  No call after init allocates.  Every call
 * taking a `stream` (a cudaStream_t; NULL = legacy default stream) is
 * asynchronous on that stream.  Calls that use one hd_ctx must be ordered on
 * one stream (the workspace is shared) and made from one host thread at a
 * time (the context keeps host-side launch state).
 *
 * Errors: every call returns an hd_status and nothing throws or aborts across
 * the ABI.  Arguments that can be checked on the host are checked before any
 * launch.  Values only the device sees (context lengths) are checked by the
 * kernels, which skip the offending sequence and record a bit in the context's
 * device error word; read and clear it with hybrid_decode_device_errors.
 *
 * Layouts (all row-major, elements):
 *   q, out           [batch][num_q_heads][head_dim]
 *   k, v (new token) [batch][num_kv_heads][head_dim]
 *   q_rot            [batch][num_q_heads][head_dim] fp32
 *   lse              [batch][num_q_heads] fp32
 *   sink             [num_q_heads] fp32
 *   gate             [batch][num_q_heads] fp32 logits
 *   cache k / v      sequence b starts at b * seq_stride; within it
 *                    [num_kv_heads][capacity][head_dim], bf16 or E4M3 codes
 *   k_scale, v_scale [num_kv_heads] fp32 (FP8 caches)
 */
#ifndef HYBRID_DECODE_H
#define HYBRID_DECODE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    HD_OK = 0,
    HD_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad enum, misaligned buffer */
    HD_ERR_UNSUPPORTED = 2,  /* a shape this library does not implement (head_dim != 256, group > 8) */
    HD_ERR_CAPACITY = 3,     /* batch > max_batch, cache capacity too small, context hint too large */
    HD_ERR_CUDA = 4,         /* a CUDA runtime/driver call or a launch failed */
    HD_ERR_STATE = 5         /* wrong layer type for the call, no device available, or
                              * the current device is not the context's device */
} hd_status;

typedef enum { HD_SLIDING = 0, HD_FULL = 1 } hd_layer_type;

/* Cache layout of sliding layers (spark_export.py, `SparkStepConfig.cache_layout`):
 * AUTO picks RING for sliding layers; full layers always append. */
typedef enum { HD_LAYOUT_AUTO = 0, HD_LAYOUT_RING = 1, HD_LAYOUT_ROLL = 2 } hd_layout;

/* Element type of every K/V cache of a context.  HD_KV_FP8_E4M3 is an
 * extension beyond the pages' bf16 step (they name FlashMLA's FP8 KV cache,
 * flashmla_sparse.py `is_fp8_kvcache`, only as prior art): entries are OCP FP8
 * E4M3 codes (torch.float8_e4m3fn bits) with one fp32 scale per kv head for K
 * and one for V (hd_kv_cache.k_scale / v_scale); a cached value is
 * code * scale.  The new entry is stored as e4m3(x / scale), x being the fp64
 * rotated key (one rounding, as for bf16) or the bf16 value, the division
 * rounded once in fp64 and the quotient rounded once to E4M3 (nearest, ties
 * to even), finite quotients beyond 448 saturating to +-448; it is scored as
 * stored.  Attention reads half the bytes of a bf16 cache. */
typedef enum { HD_KV_BF16 = 0, HD_KV_FP8_E4M3 = 1 } hd_kv_dtype;

/* Bits of the device error word (hybrid_decode_device_errors). */
enum {
    HD_DEVERR_CONTEXT_NEGATIVE = 1,  /* context[b] < 0                                     */
    HD_DEVERR_CONTEXT_CAPACITY = 2,  /* full layer: context[b] >= cache capacity            */
    HD_DEVERR_CONTEXT_PLAN = 4,      /* context[b] > max_context (table / split plan)       */
    HD_DEVERR_WAIT_TIMEOUT = 8       /* a pipeline wait gave up after its time limit        */
};

typedef struct hd_ctx hd_ctx;

/* Model shape (spark_export.py, `SparkStepConfig`), validated like its
 * `__post_init__`: num_q_heads must be a multiple of num_kv_heads, every layer
 * type must be HD_SLIDING or HD_FULL, the layout must be one of hd_layout. */
typedef struct {
    int32_t num_layers;
    const int32_t *layer_types;    /* host array [num_layers] of hd_layer_type        */
    int32_t num_q_heads;
    int32_t num_kv_heads;          /* num_q_heads / num_kv_heads <= 8                  */
    int32_t head_dim;              /* 256                                              */
    int32_t sliding_window;        /* window counting the current token (512)          */
    int32_t rotary_dim_sliding;    /* even, <= head_dim (256)                          */
    int32_t rotary_dim_full;       /* even, <= head_dim (64)                           */
    double rope_theta_sliding;     /* 1e4                                              */
    double rope_theta_full;        /* 5e6                                              */
    int32_t cache_layout;          /* hd_layout for the sliding layers                 */
    int32_t max_batch;             /* largest batch any call passes                    */
    int32_t max_context;           /* largest context (previous tokens) any call uses  */
    int32_t kv_dtype;              /* hd_kv_dtype of every cache (0 = bf16)            */
} hd_config;

/* One layer's KV cache (caller-owned device memory, of the context's
 * kv_dtype). capacity is the number of entries per (sequence, kv head):
 * window-1 for a sliding ring, window for a sliding roll window, at least
 * max_context+1 for a full layer.  seq_stride (in elements) >=
 * num_kv_heads*capacity*head_dim and a multiple of 16 bytes (8 bf16, 16 E4M3
 * elements); k and v 16-byte aligned.  k_scale / v_scale: FP8 caches only,
 * device fp32 [num_kv_heads], required there and NULL for bf16. */
typedef struct {
    void *k;
    void *v;
    int64_t seq_stride;
    int32_t capacity;
    const float *k_scale;
    const float *v_scale;
} hd_kv_cache;

/* Per-layer tensors of a whole decode step (decode_step). */
typedef struct {
    const void *q;        /* bf16 [batch][num_q_heads][head_dim], 16-byte aligned  */
    const void *k;        /* bf16 [batch][num_kv_heads][head_dim], 16-byte aligned */
    const void *v;        /* bf16 [batch][num_kv_heads][head_dim], 16-byte aligned */
    hd_kv_cache cache;
    const float *sink;    /* fp32 [num_q_heads] or NULL (no sink)                  */
    void *out;            /* bf16 [batch][num_q_heads][head_dim]                   */
    float *lse;           /* fp32 [batch][num_q_heads]                             */
    const float *gate;    /* fp32 [batch][num_q_heads] gate logits or NULL (none)  */
} hd_layer_io;

/* Pure host check of a configuration (no device use). */
hd_status hd_validate_config(const hd_config *cfg);

/* Split-K plan used for a single-layer call (pure host function, no device
 * use): keys per chunk (a power of two from 64 to 2048) and the number of
 * chunks (the grid's key dimension) for `batch` sequences of at most
 * `max_keys` scored cache keys on `num_sms` SMs.  A call on a context uses the
 * same model, bounded by the context's workspace.  decode_step's step grid
 * plans one chunk size over all its layers instead. */
hd_status hd_plan_split(int32_t batch, int32_t num_kv_heads, int32_t max_keys, int32_t num_sms,
                        int32_t *chunk_keys, int32_t *num_chunks);

/* Chunk size of a decode_step step grid (pure host function, no device use):
 * one size, a multiple of 64 keys up to 2048 (bf16) or 4096 (E4M3), for all
 * num_layers layers of `batch` sequences, layer i scoring at most max_keys[i]
 * cached keys per sequence; one_chunk (NULL: none) marks layers that take a
 * single chunk of max(chunk, max_keys[i]) keys (rolled windows).  rows: query
 * rows per kv head of the pass (group x tokens); multi_token: a pass of a
 * multi-token step.  It minimises the grid-time estimate decode_step uses (each
 * CTA's keys plus a fixed ~256 KiB-equivalent start and combine cost, per SM). */
hd_status hd_plan_step_split(int32_t num_layers, const int32_t *max_keys, const uint8_t *one_chunk,
                             int32_t batch, int32_t num_kv_heads, int32_t rows, int32_t multi_token,
                             int32_t kv_dtype, int32_t num_sms, int32_t *chunk_keys);

/* Creates a context on the current CUDA device: validates cfg (the checks of
 * spark_export.py `SparkStepConfig.__post_init__`), builds the RoPE tables for
 * positions 0..max_context -- per layer type, cos/sin of
 * position * theta^(-2i/rotary_dim) as `_angles` defines them, evaluated in
 * fp64 and stored fp32 -- and allocates the workspace sized by
 * max_batch/max_context.  Synchronous.  Errors: HD_ERR_INVALID_ARG /
 * HD_ERR_UNSUPPORTED from the config checks, HD_ERR_UNSUPPORTED on a device
 * that is not sm_103, HD_ERR_CUDA when an allocation fails (nothing is left
 * allocated then). */
hd_status hybrid_decode_init(const hd_config *cfg, hd_ctx **out_ctx);

/* Frees the context and its workspace (synchronises the device first). */
hd_status hybrid_decode_destroy(hd_ctx *ctx);

/* Rotates q (written to q_rot, fp32) and the new k for one layer, and stores
 * the new K/V entry: full layers at index context[b]; sliding ring layers into
 * the context's staging row (committed to slot context[b] mod (window-1) by
 * decode_attn_sliding after it has read the ring); sliding roll layers shift
 * their window by one when it is full and append.  (spark_export.py `_rope`,
 * `_angles`, `_Layer.forward` cache branches.) */
hd_status rope_append_kv(hd_ctx *ctx, int32_t layer, int32_t batch, const int32_t *context,
                         const void *q, const void *k, const void *v, float *q_rot,
                         hd_kv_cache cache, void *stream);

/* Attention of a sliding layer over its window (spark_export.py
 * `_Layer.forward`: the ring branch scores the cached ring and the new entry
 * as two key sets of one softmax and leaves the slot write to the runtime;
 * the roll branch scores the shifted window; the window of
 * `SparkStepConfig.cache_len` counts the current token): the ring's valid
 * slots plus the staged new entry (ring), or the rolled window (roll);
 * split-K over the keys, then an LSE combine that applies the sink
 * (flashmla_sparse.py `HYV4FlashMLASparseImpl`) and the output gate (either
 * may be NULL), writes out/lse and commits the staged ring entry to slot
 * context[b] mod (window-1).  Must follow rope_append_kv of the same layer on
 * the same stream.  Errors: HD_ERR_STATE for a full layer or a device other
 * than the context's; HD_ERR_CAPACITY when cache.capacity is not the layout's
 * (window-1 ring, window roll); contexts beyond max_context are flagged on
 * the device (HD_DEVERR_*) and give NaN out/lse for that sequence. */
hd_status decode_attn_sliding(hd_ctx *ctx, int32_t layer, int32_t batch, const int32_t *context,
                              const float *q_rot, hd_kv_cache cache, const float *sink,
                              const float *gate, void *out, float *lse, void *stream);

/* Attention of a full layer over positions 0..context[b] (spark_export.py
 * `_Layer.forward` on a full-attention layer: every cached position plus the
 * new one; `SparkStepConfig.cache_len` of a full layer is the whole context;
 * the new entry was appended at index context[b] by rope_append_kv):
 * split-K over chunks of keys sized from max_context_hint (an upper bound on
 * every context[b] of this call, <= max_context; 0 means max_context), then
 * the LSE combine with the sink (flashmla_sparse.py `HYV4FlashMLASparseImpl`)
 * and the output gate (either may be NULL).  Errors: HD_ERR_STATE for a
 * sliding layer or a device other than the context's; HD_ERR_CAPACITY when
 * the hint exceeds max_context or cache.capacity <= hint; a context[b] above
 * the hint or the capacity is flagged on the device and gives NaN out/lse. */
hd_status decode_attn_full(hd_ctx *ctx, int32_t layer, int32_t batch, const int32_t *context,
                           int32_t max_context_hint, const float *q_rot, hd_kv_cache cache,
                           const float *sink, const float *gate, void *out, float *lse, void *stream);

/* One decode step over all layers (spark_export.py `SparkDecodeStep.forward`:
 * every layer of the step with its own cache pair, the layer's type picking
 * its window, rotary table and cache layout as `SparkStepConfig.layout_for`
 * does), with the same results as rope_append_kv
 * followed by the layer's attention call for each layer in order: q is
 * rotated in the attention kernel and the new entry is rotated, scored and
 * stored (appended, or written to its ring slot after the ring was read) by
 * the combine; a roll layout's kernel reads the window, shifts it down by one
 * row once it is full and stores the new entry at its end.  `layers` is a host
 * array [num_layers].  The layers of a call are independent: by default one
 * grid runs the attention of all of them (hybrid_decode_set_step_fusion),
 * otherwise one kernel per layer, each of which may start streaming its own
 * cache while the previous layer is still running.  So within one call no
 * layer's inputs or cache may alias another layer's outputs or cache.  The
 * step waits for all earlier work in the stream.  Every layer is checked
 * before anything is launched. */
hd_status decode_step(hd_ctx *ctx, int32_t batch, const int32_t *context, int32_t max_context_hint,
                      const hd_layer_io *layers, void *stream);

/* Multi-token decode (an extension: the pages' step is one token): num_tokens
 * (1..8) new tokens per sequence at positions context[b] .. context[b] +
 * num_tokens - 1, with the same results as num_tokens decode_step calls in
 * order -- token t attends causally to its window, which holds the earlier new
 * tokens -- as in speculative verification.  Layouts gain a token index after
 * the batch index: q, out [batch][num_tokens][num_q_heads][head_dim]; k, v
 * [batch][num_tokens][num_kv_heads][head_dim]; lse, gate
 * [batch][num_tokens][num_q_heads].  The tokens of a sequence are extra query
 * rows sharing one read of the cache, up to 32 rows (bf16 caches; 16 with
 * E4M3) and 8 tokens per kv head per pass (group 4: eight tokens in one pass;
 * 32-row passes run on the tcgen05 tensor cores, see hybrid_decode_set_consumer).
 * Full layers append num_tokens entries;
 * sliding ring layers write slots (c + t) mod (window-1) after reading;
 * sliding roll layers read their window once, then drop the entries that leave
 * it (the window shifts down by that many rows) and append the num_tokens
 * entries.  HD_ERR_UNSUPPORTED for num_tokens > 1 with the CUDA-core
 * consumer; for full layers max_context_hint bounds context[b] (0 means
 * max_context - num_tokens + 1). */
hd_status decode_step_tokens(hd_ctx *ctx, int32_t batch, int32_t num_tokens, const int32_t *context,
                             int32_t max_context_hint, const hd_layer_io *layers, void *stream);

/* Layer overlap in decode_step / decode_step_tokens (default 1): a layer's
 * kernel starts reading its inputs and streaming its cache while the previous
 * layer drains, and waits for it only before its first write.  decode_step
 * takes every layer's q up front; in a model whose next q depends on this
 * layer's output only the cache prefetch part of that overlap applies.  0
 * runs every layer in full stream order (measurement, comparison). */
hd_status hybrid_decode_set_layer_overlap(hd_ctx *ctx, int32_t enable);

/* Step fusion in decode_step / decode_step_tokens (default 1): the attention of
 * all layers of a call (of a pass, with several tokens) runs as one grid --
 * up to 32 layers per grid, as many as the split-K workspace holds -- with
 * one chunk size planned over all layers, instead of one kernel per layer.
 * The results are the same.  It applies with the tensor-core consumer when no
 * layer's out, lse or cache overlaps memory of another layer of the call
 * (checked on the host); otherwise, or with 0, each layer runs its own kernel
 * (overlapping as hybrid_decode_set_layer_overlap says). */
hd_status hybrid_decode_set_step_fusion(hd_ctx *ctx, int32_t enable);

/* Chunk merge of single-layer launches (default 1): when a call's grid is
 * small enough for one CTA per SM, every chunk of a (sequence, kv head) runs in
 * one thread-block cluster (up to 16 CTAs on this part), and the chunks'
 * partials merge through distributed shared memory, each CTA finishing a slice
 * of the output; otherwise (and with 0) the last chunk to finish merges them
 * from the workspace.  The results are the same within the stated tolerance.
 * Applies to rope_append_kv's attention calls and to decode_step without step
 * fusion; step grids always merge through the workspace. */
hd_status hybrid_decode_set_cluster_combine(hd_ctx *ctx, int32_t enable);

/* Inner loop of the attention kernels (same results within the stated
 * tolerance; the default is the tensor-core one):
 *   HD_CONSUMER_CUDA_CORE     fp32 FMA with warp-shuffle reductions (one
 *                             token per sequence only);
 *   HD_CONSUMER_TENSOR_CORE   mma.sync bf16 (q split into a bf16 high and low
 *                             part) with fp32 accumulation; multi-token passes
 *                             of 32 query rows per kv head over bf16 caches
 *                             (group x tokens, e.g. 4 x 8 or 8 x 4) run on the
 *                             tcgen05 tensor cores with scores and outputs in
 *                             tensor memory, one read of the cache for the 32
 *                             rows;
 *   HD_CONSUMER_TENSOR_MEMORY as HD_CONSUMER_TENSOR_CORE, and passes of 16
 *                             rows also on tcgen05 (measured slower on GB300
 *                             for that shape; kept selectable). */
enum { HD_CONSUMER_CUDA_CORE = 0, HD_CONSUMER_TENSOR_CORE = 1, HD_CONSUMER_TENSOR_MEMORY = 2 };
hd_status hybrid_decode_set_consumer(hd_ctx *ctx, int32_t consumer);

/* Test hook for failure detection (no counterpart in the pages).  With
 * stage >= 0, the copy producer of every attention CTA stops issuing copies at
 * that pipeline stage, as if the copy were lost; the consumers' waits, bounded
 * to one second, run out, the kernel records HD_DEVERR_WAIT_TIMEOUT and
 * returns (outputs of affected sequences are then meaningless), and the
 * context stays usable.  -1 (the default) turns it off. */
hd_status hybrid_decode_inject_lost_copy(hd_ctx *ctx, int32_t stage);

/* Reads and clears the device error word (HD_DEVERR_* bits).  Synchronises
 * `stream`. */
hd_status hybrid_decode_device_errors(hd_ctx *ctx, int32_t *flags, void *stream);

/* Kernel launches issued by this context since init (host counter). */
hd_status hybrid_decode_launch_count(hd_ctx *ctx, int64_t *launches);

/* Profiling: `enable` is a mask of layer types, bit (1 << hd_layer_type):
 * HD_PROFILE_SLIDING, HD_PROFILE_FULL, both, or 0 (off), optionally with
 * HD_PROFILE_FIRST_ONLY: then only the first layer of each selected type in
 * each decode_step call is bracketed.  Attention-kernel launches of the
 * selected types are bracketed by CUDA events on their stream (up to 4096
 * launches per type between reads), and a bracketed launch does not start
 * before the previous work in the stream is complete (decode_step otherwise
 * lets a layer start streaming while the previous layer drains), so the
 * events time the kernel alone and the other layers keep overlapping.
 * With step fusion on, decode_step launches step grids instead of layer
 * kernels: HD_PROFILE_STEP brackets each step grid (up to 4096 between reads,
 * read back with layer_type HD_PROFILE_KIND_STEP); the layer-type bits then
 * bracket only layers that run their own launch.
 * hybrid_decode_profile synchronises on the events and returns, for layers of
 * the given hd_layer_type (or step grids), the summed kernel time and launch
 * count since the last read, then resets those records. */
enum {
    HD_PROFILE_SLIDING = 1 << HD_SLIDING,
    HD_PROFILE_FULL = 1 << HD_FULL,
    HD_PROFILE_FIRST_ONLY = 4,
    HD_PROFILE_STEP = 8
};
enum { HD_PROFILE_KIND_STEP = 2 };
hd_status hybrid_decode_set_profiling(hd_ctx *ctx, int32_t enable);
hd_status hybrid_decode_profile(hd_ctx *ctx, int32_t layer_type, double *total_ms, int64_t *launches);

/* Bytes of the file-scope device array that decode_attn_full_static_scratch
 * uses as its split-K scratch (64 MiB). */
#define HD_STATIC_SCRATCH_BYTES (64u << 20)

/* Full-layer attention that allocates nothing (no counterpart in the paper;
 * it exists for callers that cannot call cudaMalloc once running, such as a
 * plugin inside a runtime that pre-plans every device allocation, or a
 * serving loop where cudaMalloc/cudaFree could synchronise the device).
 * Same result as decode_attn_full (after rope_append_kv appended the new
 * entry at index context[b]; scores positions 0..context[b]), but it needs no
 * hd_ctx: the caller passes the inputs and outputs and the shape, and the
 * split-K scratch lives in one HD_STATIC_SCRATCH_BYTES file-scope device
 * array of the library (held on every GPU that uses the library until the
 * process exits).  bf16 caches only (k_scale / v_scale must be NULL).
 *   max_context  upper bound on every context[b] of this call; max_context+1
 *                <= cache.capacity.
 * Returns HD_ERR_CAPACITY, before anything is launched, when the call's
 * scratch would exceed the array (decode_attn_full_static_scratch_plan gives
 * the figure: about batch * num_q_heads * chunks * 1032 bytes, chunks =
 * ceil((max_context+1)/chunk) with chunk <= 2048).  All calls share the array
 * and it keeps the last call's contents (the tickets and the error word are
 * cleared at every call), so calls that overlap on the GPU race: order them on
 * one stream.  The first call in a CUDA context looks up the array's address
 * for that device and context; make it before any stream capture (a context
 * made again after cudaDeviceReset gets its own lookup at its first call).
 * Device-side faults of the inputs are not reported: a context[b] outside
 * [0, max_context] gives NaN out/lse for that sequence, and a pipeline wait
 * that runs out (one second) leaves that sequence's out/lse meaningless; the
 * error word that records both lives in the shared array and no call reads
 * it back. */
hd_status decode_attn_full_static_scratch(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                          const int32_t *context, int32_t max_context,
                                          const float *q_rot, hd_kv_cache cache, const float *sink,
                                          void *out, float *lse, void *stream);

/* The split plan of decode_attn_full_static_scratch and the scratch bytes it
 * needs, for `num_sms` SMs (pure host function, no device use): HD_OK when
 * the call fits the array, HD_ERR_CAPACITY when it would be refused (the
 * outputs are still written), HD_ERR_INVALID_ARG / HD_ERR_UNSUPPORTED for
 * shapes the entry point rejects.  Output pointers may be NULL. */
hd_status decode_attn_full_static_scratch_plan(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                               int32_t max_context, int32_t num_sms, int64_t *scratch_bytes,
                                               int32_t *chunk_keys, int32_t *num_chunks);

/* Measurement utility (no counterpart in the pages): one pass of a pure read
 * stream over `bytes` of the device buffer (16-byte aligned), through shared
 * memory with 1-D bulk copies, two CTAs per SM, no arithmetic; the caller
 * times it on `stream`.  Gives the read bandwidth HBM delivers on this part,
 * next to the copy figure (which counts a read and a write per byte).  Reads
 * a whole number of 32 KiB stages per CTA and may leave a tail unread. */
hd_status hybrid_decode_read_probe(const void *buffer, int64_t bytes, void *stream);

/* Static text for a status code. */
const char *hd_status_string(hd_status status);

#ifdef __cplusplus
}
#endif

#endif /* HYBRID_DECODE_H */
