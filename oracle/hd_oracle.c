/*
 * hd_oracle.c -- fp64 CPU oracle for single-token decode attention of a hybrid
 * sliding/full GQA model.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no code, header, table or constant generator with the
 * CUDA library; it is written from the sources below, in plain loops, in fp64.
 *
 * Sources (web pages; a citation is the page's file name plus the section):
 *   [spark] vllm_omni/edge/spark_export.py (vllm-omni) -- Spark-X2.5 decode step
 *   [hyv4]  vllm/models/hy_v4/nvidia/flashmla_sparse.py -- per-head attention sink
 *
 * Readings taken where the pages leave a step open (each is also listed in the
 * design notes of the repository):
 *   R1  rotary table precision: cos/sin are evaluated in fp64 from the angle
 *       position * (1 / theta^(2i/rotary_dim)) and rounded once to fp32.  [spark]
 *       `_angles` builds the same table in fp32; the fp64 angle avoids its loss
 *       of phase at long positions while keeping the stored precision.
 *   R2  the written key is bf16_rne(k1*c - k2*s) (and bf16_rne(k2*c + k1*s) for
 *       the partner dim), with k bf16, c/s the fp32 table values, the two
 *       products exact in fp64 and one fp64 rounding of the sum, then one
 *       round-to-nearest-even to bf16.  V is stored bit for bit.
 *   R3  ring slot for the token at position c is c mod (window-1); the new entry
 *       is scored from the step's own K/V and committed to its slot only after
 *       the cached keys have been scored ([spark] `_Layer.forward`, ring branch:
 *       the runtime writes the returned entry after the graph ran).
 *   R4  roll layout before step c holds positions max(0,c-window)..c-1 in order;
 *       the new entry is appended and, only once the window is full, the oldest
 *       is dropped.  (The fixed-shape export drops one entry unconditionally;
 *       the page states both layouts score the same keys, which holds only with
 *       this reading.)
 *   R5  lse is the natural-log log-sum-exp of the scaled scores, without the
 *       sink; the sink multiplies the output by exp(lse)/(exp(lse)+exp(sink))
 *       ([hyv4] HYV4FlashMLASparseImpl docstring).  A sink of -inf is no sink.
 *   R13 the optional output gate multiplies each query head's attention output
 *       by sigmoid(gate logit) after the sink ([spark] `_Layer.forward`: the
 *       attention output, viewed per head, times sigmoid(g_proj(h))); the
 *       logits are an input here (the projection lies outside the path) and
 *       do not change lse.
 *   R14 FP8 KV cache (an extension the pages name only as prior art: FlashMLA's
 *       FP8 KV cache, [hyv4] `is_fp8_kvcache`): entries are OCP FP8 E4M3 codes
 *       with one fp32 scale per kv head for K and one for V; a cached value is
 *       decode(code) * scale.  The new entry is quantised as
 *       code = e4m3(x / scale) with x the fp64 rotated key (as in R2) or the
 *       bf16 value, the division rounded once in fp64 and the result rounded
 *       once to e4m3 (nearest, ties to even), finite values beyond the largest
 *       code saturating to +-448.  The new entry is scored as stored (its
 *       dequantised value).
 *   R15 multi-token decode (the pages' step is one token; several query
 *       positions per step are an extension, as in speculative verification):
 *       T new tokens at positions c .. c+T-1 of one sequence compute exactly
 *       what T single-token steps compute in order -- token t attends
 *       causally to the layer's key set at position c+t, which holds the
 *       earlier new tokens, and the cache ends as after the T steps.
 *
 * Every function below names what pins it in the test suite (tests/).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_SLIDING 0
#define ORC_FULL 1
#define ORC_LAYOUT_RING 1
#define ORC_LAYOUT_ROLL 2

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_CAPACITY 3

/* ---------------------------------------------------------------- bf16 --- */

/* bf16 is the top half of an IEEE binary32. */
double orc_bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One round-to-nearest-even from a double to bf16 (8 significant bits,
 * binary32 exponent range).  The double is scaled so that one bf16 quantum
 * becomes 1.0, rounded to an integer with rint() (ties to even in the default
 * rounding mode), and scaled back; both scalings are exact powers of two.
 * Pinned by: tie cases built by hand, the binary32 subset against torch's
 * float->bfloat16 cast, and the half-quantum error bound on random doubles. */
uint16_t orc_f64_to_bf16(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isinf(a))
        return sign | 0x7F80;
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);            /* a = m * 2^e, m in [0.5, 1)            */
    int E = e - 1;           /* a = (2m) * 2^E, 2m in [1, 2)          */
    if (E < -126)
        E = -126;            /* bf16 subnormals share the 2^-133 quantum */
    double r = rint(ldexp(a, 7 - E)); /* quantum 2^(E-7) -> 1.0           */
    double v = ldexp(r, E - 7);
    const double bf16_max = ldexp(255.0, 127 - 7); /* (2 - 2^-7) * 2^127 */
    if (v > bf16_max)
        return sign | 0x7F80;
    float f = (float)v;      /* exact: v has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* ------------------------------------------------------ fp8 e4m3 (R14) --- */

/* OCP FP8 E4M3 ("e4m3fn"): sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; no infinities; S.1111.111 is NaN; the largest finite value is
 * 1.75 * 2^8 = 448; exponent field 0 holds the subnormals m * 2^-9.
 * Pinned by: all 256 codes against torch's float8_e4m3fn -> float32 cast. */
double orc_e4m3_to_f64(uint8_t code)
{
    int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7)
        return NAN;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return sign ? -v : v;
}

/* One round-to-nearest-even from a double to E4M3, saturating: the double is
 * scaled so that one E4M3 quantum (2^(E-3) for a value in [2^E, 2^(E+1)),
 * 2^-9 below 2^-6) becomes 1.0, rounded with rint() (ties to even) and scaled
 * back; results above 448, and infinities, become +-448; NaN stays NaN.
 * Pinned by: round trip of every finite code, brute-force nearest (ties to
 * the even code) on random and midpoint doubles, and torch's cast on binary32
 * inputs within range. */
uint8_t orc_f64_to_e4m3(double x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs(x);
    if (isinf(a))
        return sign | 0x7E;
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);
    int E = e - 1;                     /* a in [2^E, 2^(E+1)) */
    if (E < -6)
        E = -6;                        /* subnormals share the 2^-9 quantum */
    double v = ldexp(rint(ldexp(a, 3 - E)), E - 3);
    if (v > 448.0)
        return sign | 0x7E;
    if (v == 0.0)
        return sign;
    frexp(v, &e);
    E = e - 1;                         /* rounding may have moved v up one binade */
    if (E < -6)
        return sign | (uint8_t)ldexp(v, 9);               /* subnormal: m * 2^-9 */
    int mant = (int)ldexp(v, 3 - E) - 8;                   /* v = (8 + m) * 2^(E-3) */
    return sign | (uint8_t)((E + 7) << 3) | (uint8_t)mant;
}

/* ---------------------------------------------------------- rotary (R1) --- */

/* cos/sin of the rotary angles at one position, for the rotary_dim/2 pair
 * frequencies inv_i = 1 / theta^(2i / rotary_dim)  ([spark] `_angles`).  The
 * page concatenates each table with itself; the pair structure makes the
 * second copy implicit here.  Pinned by: position 0 gives (1, 0); entry 0 is
 * cos/sin(position); entry rotary_dim/4 has frequency theta^-1/2; the angle
 * addition identity across positions. */
void orc_rope_angles(int64_t position, int rotary_dim, double theta,
                     float *cos_half, float *sin_half)
{
    int half = rotary_dim / 2;
    for (int i = 0; i < half; ++i) {
        double inv = 1.0 / pow(theta, (double)(2 * i) / (double)rotary_dim);
        double ang = (double)position * inv;
        cos_half[i] = (float)cos(ang);
        sin_half[i] = (float)sin(ang);
    }
}

/* Neox-style rotation of the leading rotary_dim dims of one head vector; dims
 * at and beyond rotary_dim pass through ([spark] `_rope`: the first half x1
 * and second half x2 of the rotated span map to x*cos + (-x2, x1)*sin).
 * Pinned by: identity at position 0, bit-exact pass-through, rotation of a
 * unit vector, equality with complex multiplication z*exp(i*a), and the
 * relative-position property of the rotated dot product. */
void orc_rope_f64(const double *x, int head_dim, int rotary_dim,
                  const float *cos_half, const float *sin_half, double *y)
{
    int half = rotary_dim / 2;
    for (int i = 0; i < half; ++i) {
        double c = (double)cos_half[i], s = (double)sin_half[i];
        double x1 = x[i], x2 = x[i + half];
        y[i] = x1 * c - x2 * s;
        y[i + half] = x2 * c + x1 * s;
    }
    for (int j = rotary_dim; j < head_dim; ++j)
        y[j] = x[j];
}

/* ----------------------------------------------------------- attention --- */

/* Scaled-dot-product attention of one query over n keys, one softmax, and the
 * optional per-head sink ([spark] `_Layer.forward`: scores = q.k * 1/sqrt(d),
 * softmax over keys, weights @ values; [hyv4]: out *= exp(lse) /
 * (exp(lse) + exp(sink))).  The max is subtracted before exp only to keep the
 * fp64 exponentials finite; it cancels exactly.  lse excludes the sink (R5).
 * n == 0 leaves out = 0 and lse = -inf.
 * Pinned by: scipy softmax/logsumexp on tiny inputs, one-key closed form,
 * equal-key mean, weight sum = sigmoid(lse - sink), -inf sink = no sink. */
void orc_attend(const double *q, int head_dim, int n, const double *keys,
                const double *vals, int has_sink, double sink,
                double *out, double *lse)
{
    for (int d = 0; d < head_dim; ++d)
        out[d] = 0.0;
    if (n <= 0) {
        *lse = -INFINITY;
        return;
    }
    double scale = 1.0 / sqrt((double)head_dim);
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int d = 0; d < head_dim; ++d)
            acc += q[d] * keys[(size_t)j * head_dim + d];
        s[j] = acc * scale;
        if (s[j] > m)
            m = s[j];
    }
    double z = 0.0;
    for (int j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        z += s[j];
    }
    for (int j = 0; j < n; ++j) {
        double w = s[j] / z;
        for (int d = 0; d < head_dim; ++d)
            out[d] += w * vals[(size_t)j * head_dim + d];
    }
    *lse = m + log(z);
    if (has_sink) {
        /* exp(lse)/(exp(lse)+exp(sink)) written as 1/(1+exp(sink-lse)). */
        double f = 1.0 / (1.0 + exp(sink - *lse));
        for (int d = 0; d < head_dim; ++d)
            out[d] *= f;
    }
    free(s);
}

/* ----------------------------------------------------- cache geometry --- */

/* Entries a layer holds before the step at `context` previous tokens
 * ([spark] `SparkStepConfig.cache_len`): full layers hold every previous
 * token; a sliding window counts the current token, so a ring keeps
 * window-1 previous entries and a roll window keeps `window`.
 * Pinned by: the page's 4k-context footprint (kv_cache_bytes) and the
 * token-by-token history simulation in the tests. */
int64_t orc_cache_len(int layer_type, int layout, int window, int64_t context)
{
    if (layer_type != ORC_SLIDING)
        return context;
    int64_t keep = (layout == ORC_LAYOUT_RING) ? window - 1 : window;
    return context < keep ? context : keep;
}

/* KV footprint of the hybrid model against an all-full-attention model of the
 * same shape ([spark] `kv_cache_bytes`): one entry is a K and a V row for
 * every kv head. */
void orc_kv_cache_bytes(int num_layers, const int32_t *layer_types,
                        int sliding_layout, int window, int num_kv_heads,
                        int head_dim, int bytes_per_elem, int64_t context,
                        int64_t *hybrid, int64_t *uniform)
{
    int64_t per_entry = 2LL * num_kv_heads * head_dim * bytes_per_elem;
    int64_t entries = 0;
    for (int i = 0; i < num_layers; ++i)
        entries += orc_cache_len(layer_types[i], sliding_layout, window, context);
    *hybrid = entries * per_entry;
    *uniform = (int64_t)num_layers * context * per_entry;
}

/* ------------------------------------------------------ one decode layer --- */

#define ORC_KV_BF16 0
#define ORC_KV_FP8_E4M3 1

typedef struct {
    int32_t batch, num_q_heads, num_kv_heads, head_dim;
    int32_t layer_type;   /* ORC_SLIDING / ORC_FULL                           */
    int32_t layout;       /* sliding: ORC_LAYOUT_RING / ORC_LAYOUT_ROLL        */
    int32_t window;       /* sliding window counting the current token (512)   */
    int32_t rotary_dim;
    double rope_theta;
    int32_t capacity;     /* entries per (sequence, kv head) in the cache      */
    int64_t seq_stride;   /* elements between consecutive sequences' caches    */
    int32_t kv_dtype;     /* ORC_KV_BF16 or ORC_KV_FP8_E4M3 (R14)              */
} orc_layer;

static void load_row(const uint16_t *src, int head_dim, double *dst)
{
    for (int d = 0; d < head_dim; ++d)
        dst[d] = orc_bf16_to_f64(src[d]);
}

/* One cached K or V row in fp64: bf16 bits, or E4M3 codes times the scale. */
static void load_cached_row(const orc_layer *L, const void *cache, int64_t index, double scale,
                            double *dst)
{
    const int D = L->head_dim;
    if (L->kv_dtype == ORC_KV_FP8_E4M3) {
        const uint8_t *src = (const uint8_t *)cache + index * D;
        for (int d = 0; d < D; ++d)
            dst[d] = orc_e4m3_to_f64(src[d]) * scale;
    } else {
        load_row((const uint16_t *)cache + index * D, D, dst);
    }
}

/* One decode step of one layer ([spark] `_Layer.forward` without the
 * projections, norms, gate and MLP, which lie outside the attention path):
 * rotate q and the new k at position c = context[b], score the layer's key
 * set, apply the sink, then update the cache as the layout says (append for
 * full layers, ring slot c mod (window-1) committed after scoring, or roll
 * shift).  Query head h reads kv head h / group_size ([spark]: q is viewed as
 * (kv, group, d), so consecutive query heads share a kv head).
 *
 * gate, if not NULL, holds [B][Hq] logits of the per-head output gate (R13).
 * Outputs: out [B][Hq][D] and lse [B][Hq] in fp64; optionally the rotated
 * queries qrot [B][Hq][D] and the written keys k_written [B][Hkv][D] (bf16
 * bits, or E4M3 codes for an FP8 cache).  kcache/vcache [B] x seq_stride, each
 * sequence [Hkv][capacity][D] of bf16 bits or E4M3 codes (L->kv_dtype), are
 * updated in place; an FP8 cache takes k_scale/v_scale [Hkv] (R14).  Returns ORC_OK, or an error before touching any output
 * when an argument or a context length does not fit the layer.
 * Pinned by: the brute-force and invariant tests on the pieces above, plus
 * sliding == full at context <= window-1, ring == roll, and the multi-step
 * history simulation. */
int orc_decode_layer(const orc_layer *L, const int32_t *context,
                     const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     void *kcache, void *vcache, const float *k_scale, const float *v_scale,
                     const float *sink, const float *gate, double *out, double *lse,
                     double *qrot, void *k_written)
{
    const int B = L->batch, Hq = L->num_q_heads, Hkv = L->num_kv_heads;
    const int D = L->head_dim, rot = L->rotary_dim;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0)
        return ORC_ERR_ARG;
    const int fp8 = L->kv_dtype == ORC_KV_FP8_E4M3;
    if (!fp8 && L->kv_dtype != ORC_KV_BF16)
        return ORC_ERR_ARG;
    if (fp8 && (!k_scale || !v_scale))
        return ORC_ERR_ARG;
    const size_t esize = fp8 ? 1 : 2;   /* bytes per cache element */
    if (rot < 0 || rot > D || rot % 2 != 0)
        return ORC_ERR_ARG;
    if (L->layer_type != ORC_SLIDING && L->layer_type != ORC_FULL)
        return ORC_ERR_ARG;
    const int sliding = L->layer_type == ORC_SLIDING;
    const int ring = sliding && L->layout == ORC_LAYOUT_RING;
    const int roll = sliding && L->layout == ORC_LAYOUT_ROLL;
    if (sliding && !ring && !roll)
        return ORC_ERR_ARG;
    const int64_t need_cap = ring ? L->window - 1 : (roll ? L->window : -1);
    if (sliding && L->capacity != need_cap)
        return ORC_ERR_CAPACITY;
    if (L->seq_stride < (int64_t)Hkv * L->capacity * D)
        return ORC_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        if (context[b] < 0)
            return ORC_ERR_ARG;
        if (!sliding && context[b] >= L->capacity)
            return ORC_ERR_CAPACITY;
    }
    const int g = Hq / Hkv;
    /* One row more than any key set can hold (cache entries plus the new one). */
    const int64_t max_keys = (L->capacity > L->window ? L->capacity : L->window) + 1;

    float *cs = (float *)malloc(sizeof(float) * (size_t)(rot / 2 + 1));
    float *sn = (float *)malloc(sizeof(float) * (size_t)(rot / 2 + 1));
    double *x = (double *)malloc(sizeof(double) * D);
    double *qr = (double *)malloc(sizeof(double) * D);
    double *knew = (double *)malloc(sizeof(double) * D);
    double *keys = (double *)malloc(sizeof(double) * (size_t)max_keys * D);
    double *vals = (double *)malloc(sizeof(double) * (size_t)max_keys * D);
    uint16_t *kb = (uint16_t *)malloc(sizeof(uint16_t) * D);
    uint8_t *kq = (uint8_t *)malloc((size_t)D);   /* FP8: new K and V codes */
    uint8_t *vq = (uint8_t *)malloc((size_t)D);
    int rc = ORC_OK;

    for (int b = 0; b < B; ++b) {
        const int64_t c = context[b];
        orc_rope_angles(c, rot, L->rope_theta, cs, sn);
        for (int kv = 0; kv < Hkv; ++kv) {
            const int64_t head_off = (b * L->seq_stride + (int64_t)kv * L->capacity * D) * (int64_t)esize;
            uint8_t *kc = (uint8_t *)kcache + head_off;
            uint8_t *vc = (uint8_t *)vcache + head_off;
            const uint16_t *kin = k + ((int64_t)b * Hkv + kv) * D;
            const uint16_t *vin = v + ((int64_t)b * Hkv + kv) * D;
            const double ks = fp8 ? (double)k_scale[kv] : 1.0;
            const double vs = fp8 ? (double)v_scale[kv] : 1.0;

            /* New key: rotate in fp64, round once to bf16 (R2), or divide by
             * the scale in fp64 and round once to E4M3 (R14); V likewise. */
            load_row(kin, D, x);
            orc_rope_f64(x, D, rot, cs, sn, knew);
            for (int d = 0; d < D; ++d) {
                if (fp8) {
                    kq[d] = orc_f64_to_e4m3(knew[d] / ks);
                    vq[d] = orc_f64_to_e4m3(orc_bf16_to_f64(vin[d]) / vs);
                } else {
                    kb[d] = orc_f64_to_bf16(knew[d]);
                }
            }
            const void *knew_bits = fp8 ? (const void *)kq : (const void *)kb;
            const void *vnew_bits = fp8 ? (const void *)vq : (const void *)vin;
            if (k_written)
                memcpy((uint8_t *)k_written + ((int64_t)b * Hkv + kv) * D * (int64_t)esize, knew_bits,
                       esize * D);

            /* Key set of this step: the cached entries the layout keeps, then
             * the new entry (its own phase, stored precision). */
            int64_t n = 0;
            int64_t cached = orc_cache_len(L->layer_type, L->layout, L->window, c);
            int64_t first = 0;
            if (roll && cached == L->window)
                first = 1; /* the oldest falls off once the window is full (R4) */
            if (cached > L->capacity) {
                rc = ORC_ERR_CAPACITY;
                goto done;
            }
            for (int64_t j = first; j < cached; ++j, ++n) {
                load_cached_row(L, kc, j, ks, keys + n * D);
                load_cached_row(L, vc, j, vs, vals + n * D);
            }
            load_cached_row(L, knew_bits, 0, ks, keys + n * D);   /* scored as stored */
            load_cached_row(L, vnew_bits, 0, vs, vals + n * D);
            ++n;

            for (int hh = 0; hh < g; ++hh) {
                const int h = kv * g + hh;
                load_row(q + ((int64_t)b * Hq + h) * D, D, x);
                orc_rope_f64(x, D, rot, cs, sn, qr);
                if (qrot)
                    memcpy(qrot + ((int64_t)b * Hq + h) * D, qr, sizeof(double) * D);
                const int has_sink = sink != NULL;
                const double sk = has_sink ? (double)sink[h] : 0.0;
                double *o = out + ((int64_t)b * Hq + h) * D;
                orc_attend(qr, D, (int)n, keys, vals, has_sink, sk, o, lse + (int64_t)b * Hq + h);
                if (gate) {
                    /* sigmoid(x) = 1 / (1 + exp(-x)); exp(-inf) = 0 gives exactly 1 */
                    const double gf = 1.0 / (1.0 + exp(-(double)gate[(int64_t)b * Hq + h]));
                    for (int d = 0; d < D; ++d)
                        o[d] *= gf;
                }
            }

            /* Cache update, after scoring (R3, R4). */
            int64_t slot;
            if (ring) {
                slot = c % (L->window - 1);
            } else if (roll) {
                if (c >= L->window) {
                    memmove(kc, kc + D * esize, esize * (size_t)(L->window - 1) * D);
                    memmove(vc, vc + D * esize, esize * (size_t)(L->window - 1) * D);
                    slot = L->window - 1;
                } else {
                    slot = c;
                }
            } else {
                slot = c;
            }
            if (slot < 0 || slot >= L->capacity) {
                rc = ORC_ERR_CAPACITY;
                goto done;
            }
            memcpy(kc + slot * D * (int64_t)esize, knew_bits, esize * D);
            memcpy(vc + slot * D * (int64_t)esize, vnew_bits, esize * D);
        }
    }
done:
    free(cs); free(sn); free(x); free(qr); free(knew);
    free(keys); free(vals); free(kb); free(kq); free(vq);
    return rc;
}

/* ------------------------------------------------- multi-token decode --- */

/* T tokens per sequence in one step (R15): token t of every sequence is the
 * single-token step at context[b] + t, run in order, so each token sees the
 * entries the earlier ones stored.  Layouts: q [B][T][Hq][D], k/v
 * [B][T][Hkv][D], gate [B][T][Hq] or NULL, out [B][T][Hq][D], lse [B][T][Hq].
 * Pinned by: a brute-force causal key set built from positions (tests). */
int orc_decode_tokens(const orc_layer *L, int T, const int32_t *context,
                      const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      void *kcache, void *vcache, const float *k_scale, const float *v_scale,
                      const float *sink, const float *gate, double *out, double *lse)
{
    const int B = L->batch, Hq = L->num_q_heads, Hkv = L->num_kv_heads, D = L->head_dim;
    if (T <= 0 || B < 0)
        return ORC_ERR_ARG;
    int32_t *ctx = (int32_t *)malloc(sizeof(int32_t) * (size_t)(B + 1));
    uint16_t *qt = (uint16_t *)malloc(sizeof(uint16_t) * ((size_t)B * Hq * D + 1));
    uint16_t *kt = (uint16_t *)malloc(sizeof(uint16_t) * ((size_t)B * Hkv * D + 1));
    uint16_t *vt = (uint16_t *)malloc(sizeof(uint16_t) * ((size_t)B * Hkv * D + 1));
    float *gt = (float *)malloc(sizeof(float) * ((size_t)B * Hq + 1));
    double *ot = (double *)malloc(sizeof(double) * ((size_t)B * Hq * D + 1));
    double *lt = (double *)malloc(sizeof(double) * ((size_t)B * Hq + 1));
    int rc = ORC_OK;
    for (int t = 0; t < T && rc == ORC_OK; ++t) {
        for (int b = 0; b < B; ++b) {
            ctx[b] = context[b] + t;
            memcpy(qt + (size_t)b * Hq * D, q + ((size_t)b * T + t) * Hq * D, sizeof(uint16_t) * Hq * D);
            memcpy(kt + (size_t)b * Hkv * D, k + ((size_t)b * T + t) * Hkv * D, sizeof(uint16_t) * Hkv * D);
            memcpy(vt + (size_t)b * Hkv * D, v + ((size_t)b * T + t) * Hkv * D, sizeof(uint16_t) * Hkv * D);
            if (gate)
                memcpy(gt + (size_t)b * Hq, gate + ((size_t)b * T + t) * Hq, sizeof(float) * Hq);
        }
        rc = orc_decode_layer(L, ctx, qt, kt, vt, kcache, vcache, k_scale, v_scale, sink, gate ? gt : NULL,
                              ot, lt, NULL, NULL);
        for (int b = 0; b < B && rc == ORC_OK; ++b) {
            memcpy(out + ((size_t)b * T + t) * Hq * D, ot + (size_t)b * Hq * D, sizeof(double) * Hq * D);
            memcpy(lse + ((size_t)b * T + t) * Hq, lt + (size_t)b * Hq, sizeof(double) * Hq);
        }
    }
    free(ctx); free(qt); free(kt); free(vt); free(gt); free(ot); free(lt);
    return rc;
}
