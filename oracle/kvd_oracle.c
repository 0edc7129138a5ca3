/*
 * kvd_oracle.c -- plain, slow, obviously-correct CPU oracle for the
 * KV-cache decode-attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: it exists so that the tests, the smoke check and the
 * benchmark's CPU-baseline leg can check the CUDA library against an
 * independent restatement of the method.  It shares no code, header, table
 * or constant generator with the CUDA library.
 *
 * Sources restated here (page title, then the item on that page):
 *   [cortiq]  docs.rs cortiq-engine 0.8.49, src/cortiq_engine/kv_cache.rs
 *             (KvMode, KV_COL_WARMUP, KV_K_GROUP, LayerKvCache::quant_row,
 *              freeze_cols, append, attend, attend_group_upto, memory_bytes,
 *              evict_born, KvCache::evict, truncate_last)
 *   [rswa]    docs.rs franken_ocr 0.8.0, src/native_engine/rswa.rs
 *             (module doc, quantize_row_i8, RingCache::write_decode_step,
 *              decode_dims, decode_attention_scalar_head, decode_attention_int8,
 *              fold)
 *
 * Precision.  The quantiser is fixed by the pages to f32 arithmetic, so it
 * is written in f32 with every operation separately rounded (build with
 * -ffp-contract=off; nothing here may be contracted into an FMA).  The
 * attention itself is the plain softmax definition evaluated in f64 over
 * the dequantised cache.
 *
 * Readings taken where the pages disagree or are silent (each is listed in
 * the design notes of the repository):
 *   - ties in the quantiser round half to even (rswa quantize_row_i8 and its
 *     ties-to-even test), not half away from zero (cortiq quant_row);
 *   - the q8_2f scale keeps cortiq's floor max(absmax/127, 1e-12);
 *   - the value pass does not skip |w| < 1e-12 (cortiq attend skips them;
 *     the plain definition is used here, the difference is below 1e-7 of
 *     the output scale);
 *   - freeze: sequential p order, products and sums rounded separately,
 *     IEEE division and a correctly rounded square root.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KVO_COL_WARMUP 64 /* cortiq KV_COL_WARMUP */
#define KVO_K_GROUP 32    /* cortiq KV_K_GROUP */

enum { KVO_F32 = 0, KVO_Q8 = 1, KVO_Q8K = 2, KVO_Q8V = 3 };

/* One layer's cache for ONE sequence, as cortiq's LayerKvCache keeps it:
 * one contiguous region per KV head, rows of head_dim values.  Arrays are
 * caller-owned and sized for `cap` rows per head. */
typedef struct {
    int32_t mode;
    int32_t n_kv;
    int32_t hd;
    int32_t cap;
    const uint8_t *alive; /* [n_kv]; 0 = dead head (stores nothing) */
    int32_t seq_len;      /* rows appended (dead heads included)     */
    int32_t *head_rows;   /* [n_kv] rows actually stored per head    */
    uint8_t *kcol_set;    /* [n_kv] 1 once the K field is frozen     */
    uint8_t *vcol_set;    /* [n_kv] 1 once the V field is frozen     */
    float *k, *v;         /* [n_kv][cap][hd] (f32 components)        */
    int8_t *kq, *vq;      /* [n_kv][cap][hd] (int8 components)       */
    float *ks;            /* [n_kv][cap][ng] K scale per 32 channels */
    float *vs;            /* [n_kv][cap]     V scale per row         */
    float *kcol, *vcol;   /* [n_kv][hd]      per-channel fields      */
} kvo_cache;

static int quant_k(int mode) { return mode == KVO_Q8 || mode == KVO_Q8K; }
static int quant_v(int mode) { return mode == KVO_Q8 || mode == KVO_Q8V; }
static int n_groups(int hd) { return (hd + KVO_K_GROUP - 1) / KVO_K_GROUP; }

int kvo_k_group(void) { return KVO_K_GROUP; }
int kvo_col_warmup(void) { return KVO_COL_WARMUP; }

/* Round to nearest, ties to even, for |x| well inside the int range.
 * Written out from the definition rather than taken from the C library so
 * that the rule is visible: take the floor, compare the remainder with 1/2,
 * and break an exact tie towards the even neighbour. */
static float round_half_even(float x)
{
    float f = floorf(x);
    float rem = x - f; /* exact for |x| < 2^23 */
    if (rem > 0.5f) return f + 1.0f;
    if (rem < 0.5f) return f;
    return (fmodf(f, 2.0f) == 0.0f) ? f : f + 1.0f;
}

static int8_t to_code(float r)
{
    float t = round_half_even(r);
    if (t > 127.0f) t = 127.0f;
    if (t < -127.0f) t = -127.0f;
    return (int8_t)t;
}

/* cortiq quant_row: divide by the per-channel field (absent field = 1),
 * then per group of `group` channels: absmax, scale = max(absmax/127,
 * 1e-12), code = clamp(round(r / scale), -127, 127).  Writes n codes and
 * ceil(n/group) scales. */
void kvo_quant_row(const float *x, const float *col, int n, int group,
                   int8_t *q, float *s)
{
    float *resid = (float *)malloc(sizeof(float) * (size_t)n);
    for (int d = 0; d < n; ++d) resid[d] = col ? x[d] / col[d] : x[d];
    int gi = 0;
    for (int g0 = 0; g0 < n; g0 += group, ++gi) {
        int g1 = g0 + group < n ? g0 + group : n;
        float absmax = 0.0f;
        for (int d = g0; d < g1; ++d) {
            float a = fabsf(resid[d]);
            if (a > absmax) absmax = a;
        }
        float sc = absmax / 127.0f;
        if (sc < 1e-12f) sc = 1e-12f;
        s[gi] = sc;
        for (int d = g0; d < g1; ++d) q[d] = to_code(resid[d] / sc);
    }
    free(resid);
}

/* rswa quantize_row_i8 (the R-SWA int8 mirror): one scale per row,
 * scale = absmax/127, or 1.0 for an all-zero row; code = clamp(round(x /
 * scale)).  Kept beside quant_row because the two share the tie and
 * division rules, which the rswa tests pin with exact bit patterns. */
float kvo_quantize_row_i8(const float *x, int n, int8_t *q)
{
    float absmax = 0.0f;
    for (int d = 0; d < n; ++d) {
        float a = fabsf(x[d]);
        if (a > absmax) absmax = a;
    }
    float sc = absmax > 0.0f ? absmax / 127.0f : 1.0f;
    for (int d = 0; d < n; ++d) q[d] = to_code(x[d] / sc);
    return sc;
}

/* quantize_row_i8 on n_rows consecutive rows of n values (the int8 mirror
 * of a whole region): codes [n_rows][n], scales [n_rows]. */
void kvo_quantize_rows_i8(const float *x, long long n_rows, int n, int8_t *q, float *scales)
{
    for (long long r = 0; r < n_rows; ++r)
        scales[r] = kvo_quantize_row_i8(x + (size_t)r * (size_t)n, n, q + (size_t)r * (size_t)n);
}

/* ---- storage addressing ------------------------------------------------ */

static size_t row_off(const kvo_cache *c, int h, int p)
{
    return ((size_t)h * (size_t)c->cap + (size_t)p) * (size_t)c->hd;
}

/* cortiq freeze_cols for one component of one head: dequantise the n
 * stored rows (code * scale, one f32 product), accumulate the squares per
 * channel in row order (product, then sum, each rounded), col = max(sqrt(
 * sum / n), 1e-6), requantise every stored row against col. */
static void freeze_component(int hd, int n, int group, int8_t *q, float *s,
                             size_t q_stride_rows, float *col_out)
{
    int spp = group == hd ? 1 : n_groups(hd); /* scales per row */
    float *rows = (float *)malloc(sizeof(float) * (size_t)n * (size_t)hd);
    for (int p = 0; p < n; ++p)
        for (int d = 0; d < hd; ++d)
            rows[(size_t)p * hd + d] =
                (float)q[(size_t)p * q_stride_rows + d] * s[(size_t)p * spp + d / group];
    for (int d = 0; d < hd; ++d) col_out[d] = 0.0f;
    for (int p = 0; p < n; ++p)
        for (int d = 0; d < hd; ++d) {
            float r = rows[(size_t)p * hd + d];
            float sq = r * r;
            col_out[d] = col_out[d] + sq;
        }
    float nf = (float)n;
    for (int d = 0; d < hd; ++d) {
        float m = col_out[d] / nf;
        float r = sqrtf(m);
        col_out[d] = r > 1e-6f ? r : 1e-6f;
    }
    for (int p = 0; p < n; ++p)
        kvo_quant_row(rows + (size_t)p * hd, col_out, hd, group,
                      q + (size_t)p * q_stride_rows, s + (size_t)p * spp);
    free(rows);
}

/* The freeze trigger of cortiq append: a quantising mode, at least
 * KV_COL_WARMUP rows stored, and no field set on any head yet. */
int kvo_needs_freeze(const kvo_cache *c)
{
    if (c->mode == KVO_F32) return 0;
    if (c->seq_len < KVO_COL_WARMUP) return 0;
    for (int h = 0; h < c->n_kv; ++h)
        if (c->kcol_set[h] || c->vcol_set[h]) return 0;
    return 1;
}

/* cortiq freeze_cols over all heads (dead heads hold no rows and are left
 * without a field). */
void kvo_freeze(kvo_cache *c)
{
    int hd = c->hd, ng = n_groups(hd);
    for (int h = 0; h < c->n_kv; ++h) {
        int n = c->head_rows[h];
        if (n == 0) continue;
        if (quant_k(c->mode)) {
            freeze_component(hd, n, KVO_K_GROUP, c->kq + row_off(c, h, 0),
                             c->ks + (size_t)h * c->cap * ng, (size_t)hd,
                             c->kcol + (size_t)h * hd);
            c->kcol_set[h] = 1;
        }
        if (quant_v(c->mode)) {
            freeze_component(hd, n, hd, c->vq + row_off(c, h, 0),
                             c->vs + (size_t)h * c->cap, (size_t)hd,
                             c->vcol + (size_t)h * hd);
            c->vcol_set[h] = 1;
        }
    }
}

/* cortiq append: freeze first if due, then per live head quantise (or
 * copy) the new K and V rows; dead heads store nothing.  Returns 0, or -2
 * when the caller's capacity is exhausted. */
int kvo_append(kvo_cache *c, const float *k_new, const float *v_new)
{
    if (c->seq_len >= c->cap) return -2;
    if (kvo_needs_freeze(c)) kvo_freeze(c);
    int hd = c->hd, ng = n_groups(hd);
    for (int h = 0; h < c->n_kv; ++h) {
        if (!c->alive[h]) continue;
        int p = c->head_rows[h];
        const float *kx = k_new + (size_t)h * hd;
        const float *vx = v_new + (size_t)h * hd;
        if (quant_k(c->mode))
            kvo_quant_row(kx, c->kcol_set[h] ? c->kcol + (size_t)h * hd : NULL, hd,
                          KVO_K_GROUP, c->kq + row_off(c, h, p),
                          c->ks + ((size_t)h * c->cap + p) * ng);
        else
            memcpy(c->k + row_off(c, h, p), kx, sizeof(float) * (size_t)hd);
        if (quant_v(c->mode))
            kvo_quant_row(vx, c->vcol_set[h] ? c->vcol + (size_t)h * hd : NULL, hd, hd,
                          c->vq + row_off(c, h, p), c->vs + (size_t)h * c->cap + p);
        else
            memcpy(c->v + row_off(c, h, p), vx, sizeof(float) * (size_t)hd);
        c->head_rows[h] = p + 1;
    }
    c->seq_len += 1;
    return 0;
}

/* Dequantised (or stored f32) row p of head h: K^[d] = code * scale[d/32] *
 * kcol[d], V^[d] = code * vscale * vcol[d], fields taken as 1 before the
 * freeze.  Evaluated in f64. */
void kvo_row(const kvo_cache *c, int h, int p, int which_v, double *out)
{
    int hd = c->hd, ng = n_groups(hd);
    size_t o = row_off(c, h, p);
    if (!which_v) {
        if (quant_k(c->mode)) {
            const float *col = c->kcol_set[h] ? c->kcol + (size_t)h * hd : NULL;
            for (int d = 0; d < hd; ++d)
                out[d] = (double)c->kq[o + d] *
                         (double)c->ks[((size_t)h * c->cap + p) * ng + d / KVO_K_GROUP] *
                         (col ? (double)col[d] : 1.0);
        } else {
            for (int d = 0; d < hd; ++d) out[d] = (double)c->k[o + d];
        }
    } else {
        if (quant_v(c->mode)) {
            const float *col = c->vcol_set[h] ? c->vcol + (size_t)h * hd : NULL;
            double sv = (double)c->vs[(size_t)h * c->cap + p];
            for (int d = 0; d < hd; ++d)
                out[d] = (double)c->vq[o + d] * sv * (col ? (double)col[d] : 1.0);
        } else {
            for (int d = 0; d < hd; ++d) out[d] = (double)c->v[o + d];
        }
    }
}

/* Plain softmax attention of one query over n key/value rows supplied by a
 * row callback, in f64: s_p = scale * <q, K^_p>; m = max s; e_p = exp(s_p -
 * m); w_p = e_p / sum e; out = sum_p w_p V^_p.  probs (may be NULL) gets w. */
typedef void (*row_fn)(const void *ctx, int p, int which_v, double *out);

static void softmax_attend(const void *ctx, row_fn rows, int n, int hd,
                           const float *q, float scale, double *out, double *probs)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double *r = (double *)malloc(sizeof(double) * (size_t)hd);
    double m = -INFINITY;
    for (int p = 0; p < n; ++p) {
        rows(ctx, p, 0, r);
        double dot = 0.0;
        for (int d = 0; d < hd; ++d) dot += (double)q[d] * r[d];
        s[p] = (double)scale * dot;
        if (s[p] > m) m = s[p];
    }
    double z = 0.0;
    for (int p = 0; p < n; ++p) {
        s[p] = exp(s[p] - m);
        z += s[p];
    }
    for (int d = 0; d < hd; ++d) out[d] = 0.0;
    for (int p = 0; p < n; ++p) {
        double w = s[p] / z;
        if (probs) probs[p] = w;
        rows(ctx, p, 1, r);
        for (int d = 0; d < hd; ++d) out[d] += w * r[d];
    }
    free(r);
    free(s);
}

typedef struct {
    const kvo_cache *c;
    int h;
} head_ctx;

static void head_row(const void *ctx, int p, int which_v, double *out)
{
    const head_ctx *hc = (const head_ctx *)ctx;
    kvo_row(hc->c, hc->h, p, which_v, out);
}

/* cortiq attend: one query head over its KV head's stored rows.  Returns
 * the number of stored rows; a dead head stores none and yields zeros. */
int kvo_attend_head(const kvo_cache *c, const float *q, int kv_head, float scale,
                    double *out, double *probs)
{
    int n = c->head_rows[kv_head];
    if (n == 0) {
        for (int d = 0; d < c->hd; ++d) out[d] = 0.0;
        return 0;
    }
    head_ctx hc = {c, kv_head};
    softmax_attend(&hc, head_row, n, c->hd, q, scale, out, probs);
    return n;
}

/* cortiq attend_group: all `nheads` query heads of KV group `kv_head`; each
 * head's output is its own attend; imp (may be NULL) accumulates every
 * head's probabilities per stored row.  A dead group yields zeros and
 * leaves imp untouched. */
int kvo_attend_group(const kvo_cache *c, const float *q_group, int kv_head, int nheads,
                     float scale, double *out, double *imp)
{
    int hd = c->hd, n = c->head_rows[kv_head];
    if (n == 0) {
        for (int i = 0; i < nheads * hd; ++i) out[i] = 0.0;
        return 0;
    }
    double *probs = (double *)malloc(sizeof(double) * (size_t)n);
    head_ctx hc = {c, kv_head};
    for (int h = 0; h < nheads; ++h) {
        softmax_attend(&hc, head_row, n, hd, q_group + (size_t)h * hd, scale,
                       out + (size_t)h * hd, probs);
        if (imp)
            for (int p = 0; p < n; ++p) imp[p] += probs[p];
    }
    free(probs);
    return n;
}

/* The decode of many sequences at once, for timing the oracle on every host
 * core: the (sequence, query head) pairs are independent, so they are shared
 * among `threads` OpenMP threads (0 = the runtime's default).  Each pair runs
 * exactly the serial code above -- kvo_attend_group for one head -- with its
 * probabilities kept in a buffer of its own; the per-row masses are then
 * added into imp[i] sequence by sequence in ascending head order, the order
 * the serial group loop adds them, so the result is bitwise the serial one
 * whatever the thread count.  caches[i], qs[i] ([n_q][hd] f32) and outs[i]
 * ([n_q][hd] f64) describe sequence i; imps (NULL, or NULL entries) skips imp.
 * Returns the number of threads that ran, or -1 if a buffer could not be
 * allocated (nothing is written then). */
int kvo_decode_many(const kvo_cache *const *caches, int n_seq, const float *const *qs, int n_q,
                    float scale, double *const *outs, double *const *imps, int threads)
{
    long long n_pairs = (long long)n_seq * n_q;
    double **probs = (double **)calloc((size_t)(n_pairs > 0 ? n_pairs : 1), sizeof(double *));
    if (!probs) return -1;
    int fail = 0;
    for (long long t = 0; t < n_pairs && !fail; ++t) {
        int i = (int)(t / n_q);
        if (imps && imps[i]) {
            probs[t] = (double *)calloc((size_t)(caches[i]->cap > 0 ? caches[i]->cap : 1), sizeof(double));
            if (!probs[t]) fail = 1;
        }
    }
    int used = 1;
    if (!fail) {
#ifdef _OPENMP
        if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads)
#endif
        for (long long t = 0; t < n_pairs; ++t) {
            int i = (int)(t / n_q), h = (int)(t % n_q);
            const kvo_cache *c = caches[i];
            int hpk = n_q / c->n_kv;
            kvo_attend_group(c, qs[i] + (size_t)h * c->hd, h / hpk, 1, scale,
                             outs[i] + (size_t)h * c->hd, probs[t]);
#ifdef _OPENMP
            if (t == 0) used = omp_get_num_threads();
#endif
        }
        for (int i = 0; i < n_seq && imps; ++i) {
            if (!imps[i]) continue;
            for (int h = 0; h < n_q; ++h) {
                const kvo_cache *c = caches[i];
                int n = c->head_rows[h / (n_q / c->n_kv)];
                const double *pr = probs[(long long)i * n_q + h];
                for (int p = 0; p < n; ++p) imps[i][p] += pr[p];
            }
        }
    }
    for (long long t = 0; t < n_pairs; ++t) free(probs[t]);
    free(probs);
    return fail ? -1 : used;
}

/* cortiq attend_group_upto with its four options, in f64:
 *   - upto >= 0 limits the stored rows to min(stored, upto) (the page's causal
 *     limit: a query at position upto - 1 sees rows [0, upto)); upto < 0 = all;
 *   - only rows [first, stored) are scored, first clamped to stored - 1 (the
 *     earliest visible position; sliding-window layers pass stored - window);
 *     earlier rows have probability 0 and their imp entries are untouched;
 *   - softcap > 0: every computed score (scale * <q, K^_p>) becomes
 *     softcap * tanh(score / softcap) before the softmax (Gemma-2 logit
 *     soft-capping); a sink is not a score and is not capped;
 *   - sinks (NULL = none): one logit per head joins the softmax maximum and
 *     adds exp(sink - max) to the denominator; it has no value row (the same
 *     as appending a value-less column).
 * out = sum_p w_p V^_p with w_p = exp(s_p - m) / (sum_q exp(s_q - m) +
 * [exp(z - m)]), m = max(max_p s_p, [z]); imp[p] += w_p over the heads.  A
 * dead or empty group yields zeros and leaves imp untouched. */
int kvo_attend_group_ex(const kvo_cache *c, const float *q_group, int kv_head, int nheads,
                        float scale, int first, float softcap, long long upto,
                        const float *sinks, double *out, double *imp)
{
    int hd = c->hd, stored = c->head_rows[kv_head];
    /* upto: attend the first min(stored, upto) rows only (the page's causal
     * limit; a negative value means none) */
    if (upto >= 0 && upto < stored) stored = (int)upto;
    if (stored == 0) {
        for (int i = 0; i < nheads * hd; ++i) out[i] = 0.0;
        return 0;
    }
    if (first > stored - 1) first = stored - 1;
    if (first < 0) first = 0;
    int span = stored - first;
    double *s = (double *)malloc(sizeof(double) * (size_t)span);
    double *r = (double *)malloc(sizeof(double) * (size_t)hd);
    for (int h = 0; h < nheads; ++h) {
        const float *q = q_group + (size_t)h * hd;
        double *o = out + (size_t)h * hd;
        double m = -INFINITY;
        for (int p = first; p < stored; ++p) {
            kvo_row(c, kv_head, p, 0, r);
            double dot = 0.0;
            for (int d = 0; d < hd; ++d) dot += (double)q[d] * r[d];
            double v = (double)scale * dot;
            if (softcap > 0.0f) v = (double)softcap * tanh(v / (double)softcap);
            s[p - first] = v;
            if (v > m) m = v;
        }
        if (sinks && (double)sinks[h] > m) m = (double)sinks[h];
        double z = 0.0;
        for (int i = 0; i < span; ++i) {
            s[i] = exp(s[i] - m);
            z += s[i];
        }
        if (sinks) z += exp((double)sinks[h] - m);
        for (int d = 0; d < hd; ++d) o[d] = 0.0;
        for (int p = first; p < stored; ++p) {
            double w = s[p - first] / z;
            if (imp) imp[p] += w;
            kvo_row(c, kv_head, p, 1, r);
            for (int d = 0; d < hd; ++d) o[d] += w * r[d];
        }
    }
    free(r);
    free(s);
    return stored;
}

/* cortiq memory_bytes restricted to the stored K/V state: every f32
 * (rows, scales, fields) counts 4 bytes, every int8 code 1 byte. */
long long kvo_memory_bytes(const kvo_cache *c)
{
    long long floats = 0, bytes = 0;
    int hd = c->hd, ng = n_groups(hd);
    for (int h = 0; h < c->n_kv; ++h) {
        long long n = c->head_rows[h];
        if (quant_k(c->mode)) {
            bytes += n * hd;
            floats += n * ng;
        } else {
            floats += n * hd;
        }
        if (quant_v(c->mode)) {
            bytes += n * hd;
            floats += n;
        } else {
            floats += n * hd;
        }
        if (c->kcol_set[h]) floats += hd;
        if (c->vcol_set[h]) floats += hd;
    }
    return floats * 4 + bytes;
}

/* ---- R-SWA ------------------------------------------------------------- */

/* ---- cortiq LayerKvCache::evict_born ------------------------------------ */

typedef struct {
    float imp;
    int pos;
} born_item;

/* Highest accumulated mass first; equal mass keeps the lower position first
 * (the page orders the middle positions with a stable sort of the ascending
 * list, so this total order gives the same sequence; NaN mass is outside
 * the contract). */
static int born_cmp(const void *a, const void *b)
{
    const born_item *x = (const born_item *)a, *y = (const born_item *)b;
    if (x->imp > y->imp) return -1;
    if (x->imp < y->imp) return 1;
    return (x->pos > y->pos) - (x->pos < y->pos);
}

static void gather_rows(void *base, size_t row_bytes, const int *kept, int n)
{
    /* kept ascends and kept[j] >= j, so copying j = 0, 1, ... in order never
     * reads a row that an earlier step overwrote */
    char *b = (char *)base;
    for (int j = 0; j < n; ++j)
        if (kept[j] != j) memmove(b + (size_t)j * row_bytes, b + (size_t)kept[j] * row_bytes, row_bytes);
}

/* cortiq evict_born for one sequence, with imp its accumulated mass per
 * stored row: when more than keep_last rows are stored, keep the first
 * min(sink, keep_last) rows (attention sinks), the last min(recent,
 * keep_last - sinks) rows, and fill the rest of the budget with the middle
 * rows of highest mass; then gather the kept rows, in row order, in every
 * storage of every live head independently (f32 K and V, int8 codes with
 * their scales) and in imp.  Returns the rows kept, -1 for a negative
 * argument. */
int kvo_evict_born(kvo_cache *c, float *imp, int keep_last, int sink, int recent)
{
    if (keep_last < 0 || sink < 0 || recent < 0) return -1;
    const int stored = c->seq_len;
    if (stored <= keep_last) return stored;
    const int sink_n = sink < keep_last ? sink : keep_last;
    const int recent_n = recent < keep_last - sink_n ? recent : keep_last - sink_n;
    unsigned char *keep = (unsigned char *)calloc((size_t)stored, 1);
    for (int p = 0; p < sink_n; ++p) keep[p] = 1;
    for (int p = stored - recent_n; p < stored; ++p) keep[p] = 1;
    int budget = keep_last - sink_n - recent_n;
    born_item *order = (born_item *)malloc(sizeof(born_item) * (size_t)stored);
    int m = 0;
    for (int p = 0; p < stored; ++p)
        if (!keep[p]) {
            order[m].imp = imp[p];
            order[m].pos = p;
            ++m;
        }
    qsort(order, (size_t)m, sizeof(born_item), born_cmp);
    for (int i = 0; i < m && budget > 0; ++i, --budget) keep[order[i].pos] = 1;
    int *kept = (int *)malloc(sizeof(int) * (size_t)stored);
    int n = 0;
    for (int p = 0; p < stored; ++p)
        if (keep[p]) kept[n++] = p;
    const int hd = c->hd, ng = n_groups(hd);
    for (int h = 0; h < c->n_kv; ++h) {
        if (!c->alive[h]) continue;
        const size_t base = (size_t)h * (size_t)c->cap;
        if (c->k) gather_rows(c->k + base * hd, sizeof(float) * (size_t)hd, kept, n);
        if (c->v) gather_rows(c->v + base * hd, sizeof(float) * (size_t)hd, kept, n);
        if (c->kq) {
            gather_rows(c->kq + base * hd, (size_t)hd, kept, n);
            gather_rows(c->ks + base * ng, sizeof(float) * (size_t)ng, kept, n);
        }
        if (c->vq) {
            gather_rows(c->vq + base * hd, (size_t)hd, kept, n);
            gather_rows(c->vs + base, sizeof(float), kept, n);
        }
        c->head_rows[h] = n;
    }
    gather_rows(imp, sizeof(float), kept, n);
    /* the page truncates imp to the kept rows and each later append pushes a
     * zero; in this flat buffer the dropped rows' entries are cleared */
    for (int p = n; p < stored; ++p) imp[p] = 0.0f;
    c->seq_len = n;
    free(kept);
    free(order);
    free(keep);
    return n;
}

/* cortiq LayerKvCache::truncate_last: drop the last min(n_drop, stored)
 * rows of every storage and of imp (speculative-decode reject).  The rows'
 * bytes stay where they are (nothing reads past the length); their imp
 * entries are cleared so that rows appended later start from zero mass, as
 * each appended row does on the page.  Returns the new length. */
int kvo_truncate_last(kvo_cache *c, float *imp, int n_drop)
{
    if (n_drop < 0) return -1;
    const int d = n_drop < c->seq_len ? n_drop : c->seq_len;
    const int n = c->seq_len - d;
    for (int h = 0; h < c->n_kv; ++h)
        if (c->alive[h]) c->head_rows[h] = n;
    if (imp)
        for (int p = n; p < c->seq_len; ++p) imp[p] = 0.0f;
    c->seq_len = n;
    return n;
}

/* rswa write_decode_step for one stream: warm-up appends at ring_len and
 * sets ring_pos = ring_len % W; steady state overwrites ring_pos and
 * advances it modulo W.  Layout [H][W][hd].  Returns the slot, or -3 when
 * no prefill has been recorded (prefill_recorded == 0). */
int kvo_rswa_write(int H, int hd, int W, float *ring_k, float *ring_v, const float *k,
                   const float *v, int prefill_recorded, int32_t *ring_len, int32_t *ring_pos)
{
    if (!prefill_recorded) return -3;
    int slot;
    if (*ring_len < W) {
        slot = *ring_len;
        *ring_len += 1;
        *ring_pos = *ring_len % W;
    } else {
        slot = *ring_pos;
        *ring_pos = (*ring_pos + 1) % W;
    }
    for (int h = 0; h < H; ++h) {
        memcpy(ring_k + ((size_t)h * W + slot) * hd, k + (size_t)h * hd, sizeof(float) * (size_t)hd);
        memcpy(ring_v + ((size_t)h * W + slot) * hd, v + (size_t)h * hd, sizeof(float) * (size_t)hd);
    }
    return slot;
}

typedef struct {
    const float *ref_k, *ref_v, *ring_k, *ring_v;
    int prefill_len, hd;
} rswa_ctx;

static void rswa_row(const void *ctx, int p, int which_v, double *out)
{
    const rswa_ctx *r = (const rswa_ctx *)ctx;
    const float *src;
    if (p < r->prefill_len)
        src = (which_v ? r->ref_v : r->ref_k) + (size_t)p * r->hd;
    else
        src = (which_v ? r->ring_v : r->ring_k) + (size_t)(p - r->prefill_len) * r->hd;
    for (int d = 0; d < r->hd; ++d) out[d] = (double)src[d];
}

/* rswa decode_attention for one stream: per head, keys = reference rows
 * [0, prefill_len) followed by ring rows [0, ring_len), no mask, softmax
 * over the union.  Reference layout [H][ref_cap][hd], ring [H][W][hd].
 * Returns 0, -3 if no prefill was recorded (prefill_len < 0), -4 for an
 * empty key set. */
int kvo_rswa_decode(int H, int hd, const float *q, const float *ref_k, const float *ref_v,
                    long long ref_cap, int prefill_len, const float *ring_k, const float *ring_v,
                    int W, int ring_len, float scale, double *out)
{
    if (prefill_len < 0) return -3;
    if (prefill_len + ring_len == 0) return -4;
    for (int h = 0; h < H; ++h) {
        rswa_ctx rc = {ref_k + (size_t)h * ref_cap * hd, ref_v + (size_t)h * ref_cap * hd,
                       ring_k + (size_t)h * W * hd, ring_v + (size_t)h * W * hd,
                       prefill_len, hd};
        softmax_attend(&rc, rswa_row, prefill_len + ring_len, hd, q + (size_t)h * hd, scale,
                       out + (size_t)h * hd, NULL);
    }
    return 0;
}

/* rswa decode_attention_int8 for one stream, over the int8 mirror only:
 * per head, q is quantised per row (quantize_row_i8, giving codes and
 * qscale); each key row's score is the exact integer dot of the codes
 * times qscale times the row's K scale times `scale`; softmax over the
 * reference rows followed by the ring rows; the output is the softmax-
 * weighted sum of the dequantised V rows (code times the row's V scale).
 * Codes [H][rows][hd], scales [H][rows] for rows = ref_cap (reference) and
 * W (ring).  The integer dot is exact (its bound is 127 * 127 * hd); the
 * products and the softmax are evaluated in f64.  Returns 0, -3 with no
 * prefill (prefill_len < 0), -4 for an empty key set. */
int kvo_rswa_decode_i8(int H, int hd, const float *q, const int8_t *ref_k8, const float *ref_ks,
                       const int8_t *ref_v8, const float *ref_vs, long long ref_cap,
                       int prefill_len, const int8_t *ring_k8, const float *ring_ks,
                       const int8_t *ring_v8, const float *ring_vs, int W, int ring_len,
                       float scale, double *out)
{
    if (prefill_len < 0) return -3;
    const int n = prefill_len + ring_len;
    if (n == 0) return -4;
    int8_t *qc = (int8_t *)malloc((size_t)hd);
    double *w = (double *)malloc(sizeof(double) * (size_t)n);
    for (int h = 0; h < H; ++h) {
        const float qscale = kvo_quantize_row_i8(q + (size_t)h * hd, hd, qc);
        double m = -INFINITY;
        for (int p = 0; p < n; ++p) {
            const int8_t *k;
            float ks;
            if (p < prefill_len) {
                k = ref_k8 + ((size_t)h * (size_t)ref_cap + (size_t)p) * (size_t)hd;
                ks = ref_ks[(size_t)h * (size_t)ref_cap + (size_t)p];
            } else {
                k = ring_k8 + ((size_t)h * (size_t)W + (size_t)(p - prefill_len)) * (size_t)hd;
                ks = ring_ks[(size_t)h * (size_t)W + (size_t)(p - prefill_len)];
            }
            long long dot = 0;
            for (int d = 0; d < hd; ++d) dot += (long long)qc[d] * (long long)k[d];
            w[p] = (double)dot * (double)qscale * (double)ks * (double)scale;
            if (w[p] > m) m = w[p];
        }
        double den = 0.0;
        for (int p = 0; p < n; ++p) {
            w[p] = exp(w[p] - m);
            den += w[p];
        }
        double *o = out + (size_t)h * hd;
        for (int d = 0; d < hd; ++d) o[d] = 0.0;
        for (int p = 0; p < n; ++p) {
            const int8_t *v;
            float vs;
            if (p < prefill_len) {
                v = ref_v8 + ((size_t)h * (size_t)ref_cap + (size_t)p) * (size_t)hd;
                vs = ref_vs[(size_t)h * (size_t)ref_cap + (size_t)p];
            } else {
                v = ring_v8 + ((size_t)h * (size_t)W + (size_t)(p - prefill_len)) * (size_t)hd;
                vs = ring_vs[(size_t)h * (size_t)W + (size_t)(p - prefill_len)];
            }
            for (int d = 0; d < hd; ++d) o[d] += w[p] * (double)vs * (double)v[d];
        }
        for (int d = 0; d < hd; ++d) o[d] /= den;
    }
    free(w);
    free(qc);
    return 0;
}

/* rswa fold, the streaming form of the same softmax, kept so that a test
 * can show the two-pass definition above and the online recurrence agree:
 * per key, if the score beats the running max, scale the running sum and
 * accumulator by exp(old - new) (0 when the old max is -inf); then add
 * w = exp(score - max).  f32, in the page's order, for one head. */
void kvo_online_head(int n, int hd, const float *q, const float *keys, const float *vals,
                     float scale, float *out)
{
    float run_max = -INFINITY, run_den = 0.0f;
    float *acc = (float *)calloc((size_t)hd, sizeof(float));
    for (int p = 0; p < n; ++p) {
        float dot = 0.0f;
        for (int d = 0; d < hd; ++d) dot = dot + q[d] * keys[(size_t)p * hd + d];
        float score = dot * scale;
        if (score > run_max) {
            float corr = isinf(run_max) ? 0.0f : expf(run_max - score);
            run_den = run_den * corr;
            for (int d = 0; d < hd; ++d) acc[d] = acc[d] * corr;
            run_max = score;
        }
        float w = expf(score - run_max);
        run_den = run_den + w;
        for (int d = 0; d < hd; ++d) acc[d] = acc[d] + w * vals[(size_t)p * hd + d];
    }
    float inv = run_den > 0.0f ? 1.0f / run_den : 0.0f;
    for (int d = 0; d < hd; ++d) out[d] = acc[d] * inv;
    free(acc);
}
