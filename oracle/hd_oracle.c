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

typedef struct {
    int32_t batch, num_q_heads, num_kv_heads, head_dim;
    int32_t layer_type;   /* ORC_SLIDING / ORC_FULL                           */
    int32_t layout;       /* sliding: ORC_LAYOUT_RING / ORC_LAYOUT_ROLL        */
    int32_t window;       /* sliding window counting the current token (512)   */
    int32_t rotary_dim;
    double rope_theta;
    int32_t capacity;     /* entries per (sequence, kv head) in the cache      */
    int64_t seq_stride;   /* elements between consecutive sequences' caches    */
} orc_layer;

static void load_row(const uint16_t *src, int head_dim, double *dst)
{
    for (int d = 0; d < head_dim; ++d)
        dst[d] = orc_bf16_to_f64(src[d]);
}

/* One decode step of one layer ([spark] `_Layer.forward` without the
 * projections, norms, gate and MLP, which lie outside the attention path):
 * rotate q and the new k at position c = context[b], score the layer's key
 * set, apply the sink, then update the cache as the layout says (append for
 * full layers, ring slot c mod (window-1) committed after scoring, or roll
 * shift).  Query head h reads kv head h / group_size ([spark]: q is viewed as
 * (kv, group, d), so consecutive query heads share a kv head).
 *
 * gate, if not NULL, holds [B][Hq] logits of the per-head output gate (R6).
 * Outputs: out [B][Hq][D] and lse [B][Hq] in fp64; optionally the rotated
 * queries qrot [B][Hq][D] and the written keys k_written [B][Hkv][D] (bf16).
 * kcache/vcache [B] x seq_stride, each sequence [Hkv][capacity][D] bf16, are
 * updated in place.  Returns ORC_OK, or an error before touching any output
 * when an argument or a context length does not fit the layer.
 * Pinned by: the brute-force and invariant tests on the pieces above, plus
 * sliding == full at context <= window-1, ring == roll, and the multi-step
 * history simulation. */
int orc_decode_layer(const orc_layer *L, const int32_t *context,
                     const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     uint16_t *kcache, uint16_t *vcache, const float *sink,
                     const float *gate, double *out, double *lse, double *qrot,
                     uint16_t *k_written)
{
    const int B = L->batch, Hq = L->num_q_heads, Hkv = L->num_kv_heads;
    const int D = L->head_dim, rot = L->rotary_dim;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0)
        return ORC_ERR_ARG;
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
    int rc = ORC_OK;

    for (int b = 0; b < B; ++b) {
        const int64_t c = context[b];
        orc_rope_angles(c, rot, L->rope_theta, cs, sn);
        for (int kv = 0; kv < Hkv; ++kv) {
            uint16_t *kc = kcache + b * L->seq_stride + (int64_t)kv * L->capacity * D;
            uint16_t *vc = vcache + b * L->seq_stride + (int64_t)kv * L->capacity * D;
            const uint16_t *kin = k + ((int64_t)b * Hkv + kv) * D;
            const uint16_t *vin = v + ((int64_t)b * Hkv + kv) * D;

            /* New key: rotate in fp64, round once to bf16 (R2). */
            load_row(kin, D, x);
            orc_rope_f64(x, D, rot, cs, sn, knew);
            for (int d = 0; d < D; ++d)
                kb[d] = orc_f64_to_bf16(knew[d]);
            if (k_written)
                memcpy(k_written + ((int64_t)b * Hkv + kv) * D, kb, sizeof(uint16_t) * D);

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
                load_row(kc + j * D, D, keys + n * D);
                load_row(vc + j * D, D, vals + n * D);
            }
            load_row(kb, D, keys + n * D);
            load_row(vin, D, vals + n * D);
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
                    memmove(kc, kc + D, sizeof(uint16_t) * (size_t)(L->window - 1) * D);
                    memmove(vc, vc + D, sizeof(uint16_t) * (size_t)(L->window - 1) * D);
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
            memcpy(kc + slot * D, kb, sizeof(uint16_t) * D);
            memcpy(vc + slot * D, vin, sizeof(uint16_t) * D);
        }
    }
done:
    free(cs); free(sn); free(x); free(qr); free(knew);
    free(keys); free(vals); free(kb);
    return rc;
}
