/*
 * fp64 CPU oracle for the Gemma-4-31B decode-step attention core ("attn.core").
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * What it computes (gemma-4-31B Model Spec, "Compute-graph nodes" table,
 * rows `attn.core` / slidingDecodeGQA and `attn.core` / decodeGQA):
 *
 *   o[b,h] = sum_{s in range(b)} softmax_s( 1 * <q[b,h], k[b,s,h/g]> ) * v[b,s,h/g]
 *
 * with g = H / KVH query heads per KV head (2 for sliding layers, 8 for global
 * layers) and attention scale exactly 1.  The attended range follows the masks
 * of the "Gemma 4 31B-it Text Architecture" page, "Compact form", with the new
 * token's K/V
 * appended before attention, so the query position is t = L_b - 1 (full layers
 * attend to every s with s <= t, sliding layers to s in the half-open interval
 * (t - 1024, t]):
 *
 *   window == 0 : s in [0, L_b)
 *   window  > 0 : s in [max(0, L_b - window), L_b)
 *
 * Per (b, h) the oracle follows the plain definition, in double precision, over
 * the exact real values of the bf16 inputs:
 *   1. score_s = sum_d q[b,h,d] * k[b,s,kvh,d]           (scale 1)
 *   2. m       = max_s score_s
 *   3. e_s     = exp(score_s - m)
 *   4. l       = sum_s e_s
 *   5. o[b,h,d] = (sum_s e_s * v[b,s,kvh,d]) / l
 * The compact form fixes the softmax precision at fp32 or better; the oracle
 * computes the exact result up to fp64 rounding.
 * An empty range (L_b == 0) gives o = 0 (the empty sum).
 *
 * Inputs are bf16 bit patterns (uint16).  A bf16 value is the upper half of an
 * IEEE binary32, so widening is exact.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)

/* Exact widening of a bf16 bit pattern: the 16 bits are the high half of a
 * binary32 value. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Attended range of sequence b (Compact form masks, append-before-attend). */
static void attended_range(int64_t L, int window, int64_t *lo, int64_t *hi)
{
    *hi = L;
    *lo = (window > 0 && L > window) ? L - window : 0;
}

/*
 * Softmax-weighted sum over an explicit list of key/value rows.
 *   q_row : D doubles
 *   k_row(j), v_row(j) : pointers to D bf16 values of the j-th attended key/value
 *   n     : number of attended rows
 *   scores: scratch of n doubles
 *   out   : D doubles
 * Steps 1-5 of the definition above, one after the other.
 */
typedef const uint16_t *(*row_fn)(const void *ctx, int64_t j);

static void attend(const double *q_row, int D, int64_t n, row_fn k_row, row_fn v_row,
                   const void *ctx, double *scores, double *out)
{
    int d;
    int64_t j;
    for (d = 0; d < D; ++d) out[d] = 0.0;
    if (n <= 0) return; /* empty sum */

    /* 1. scores, scale 1 */
    for (j = 0; j < n; ++j) {
        const uint16_t *kr = k_row(ctx, j);
        double s = 0.0;
        for (d = 0; d < D; ++d) s += q_row[d] * bf16_bits_to_double(kr[d]);
        scores[j] = s;
    }
    /* 2. max */
    double m = scores[0];
    for (j = 1; j < n; ++j)
        if (scores[j] > m) m = scores[j];
    /* 3. exponentials, 4. normaliser */
    double l = 0.0;
    for (j = 0; j < n; ++j) {
        scores[j] = exp(scores[j] - m);
        l += scores[j];
    }
    /* 5. weighted sum of values, divided by the normaliser */
    for (j = 0; j < n; ++j) {
        const uint16_t *vr = v_row(ctx, j);
        const double e = scores[j];
        for (d = 0; d < D; ++d) out[d] += e * bf16_bits_to_double(vr[d]);
    }
    for (d = 0; d < D; ++d) out[d] /= l;
}

/* ---- contiguous cache: k, v are [B, S, KVH, D] holding positions [pos_base, pos_base+S) ---- */
typedef struct {
    const uint16_t *k, *v;
    int64_t b, kvh, lo, pos_base, S;
    int KVH, D;
} contig_ctx;

static const uint16_t *contig_k(const void *c, int64_t j)
{
    const contig_ctx *x = (const contig_ctx *)c;
    int64_t s = x->lo + j - x->pos_base;
    return x->k + ((x->b * x->S + s) * x->KVH + x->kvh) * x->D;
}
static const uint16_t *contig_v(const void *c, int64_t j)
{
    const contig_ctx *x = (const contig_ctx *)c;
    int64_t s = x->lo + j - x->pos_base;
    return x->v + ((x->b * x->S + s) * x->KVH + x->kvh) * x->D;
}

/*
 * q:        [B, H, D] bf16 bits
 * k, v:     [B, S, KVH, D] bf16 bits; row s of the array is position pos_base + s
 * seq_lens: [B] absolute lengths, 0 <= L_b, and every attended position must lie
 *           in [pos_base, pos_base + S)
 * window:   0 = full history (decodeGQA); > 0 = the last `window` positions
 * out:      [B, H, D] doubles
 * nthreads: OpenMP threads (<= 0: the runtime default)
 * Returns 0, or a negative code for arguments outside the definition.
 */
int oracle_gqa_decode_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          const int32_t *seq_lens, int B, int S, int H, int KVH, int D,
                          int window, int64_t pos_base, int nthreads, double *out)
{
    int b;
    if (B < 0 || S < 0 || H <= 0 || KVH <= 0 || D <= 0 || window < 0) return ORACLE_EINVAL;
    if (H % KVH != 0) return ORACLE_EINVAL;
    for (b = 0; b < B; ++b) {
        int64_t lo, hi;
        if (seq_lens[b] < 0) return ORACLE_EINVAL;
        attended_range(seq_lens[b], window, &lo, &hi);
        if (hi > lo && (lo < pos_base || hi > pos_base + S)) return ORACLE_EINVAL;
    }
    const int g = H / KVH;
    const int64_t pairs = (int64_t)B * H;
    int64_t max_n = 1;
    for (b = 0; b < B; ++b) {
        int64_t lo, hi;
        attended_range(seq_lens[b], window, &lo, &hi);
        if (hi - lo > max_n) max_n = hi - lo;
    }
    int err = ORACLE_OK;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#endif
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)max_n);
        double *q_row = (double *)malloc(sizeof(double) * (size_t)D);
        const int have_scratch = scores != NULL && q_row != NULL;
        int64_t p;
        /* every thread reaches the work-sharing loop (it ends in a barrier) */
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (p = 0; p < pairs; ++p) {
            if (!have_scratch) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                err = ORACLE_ENOMEM;
                continue;
            }
            {
                const int64_t bb = p / H, h = p % H;
                int64_t lo, hi;
                int d;
                attended_range(seq_lens[bb], window, &lo, &hi);
                for (d = 0; d < D; ++d) q_row[d] = bf16_bits_to_double(q[(bb * H + h) * D + d]);
                contig_ctx c = {k, v, bb, h / g, lo, pos_base, S, KVH, D};
                attend(q_row, D, hi - lo, contig_k, contig_v, &c, scores, out + (bb * H + h) * D);
            }
        }
        free(scores);
        free(q_row);
    }
    (void)nthreads;
    return err;
}

/* ---- paged cache: pools [P, page_size, KVH, D]; position s of sequence b lives at
 *      page block_table[b][s / page_size], slot s % page_size ---- */
typedef struct {
    const uint16_t *k, *v;
    const int32_t *bt_row;
    int64_t kvh, lo;
    int page_size, KVH, D;
} paged_ctx;

static const uint16_t *paged_row(const uint16_t *pool, const paged_ctx *x, int64_t j)
{
    int64_t s = x->lo + j;
    int64_t page = x->bt_row[s / x->page_size];
    int64_t slot = s % x->page_size;
    return pool + ((page * x->page_size + slot) * x->KVH + x->kvh) * x->D;
}
static const uint16_t *paged_k(const void *c, int64_t j)
{
    const paged_ctx *x = (const paged_ctx *)c;
    return paged_row(x->k, x, j);
}
static const uint16_t *paged_v(const void *c, int64_t j)
{
    const paged_ctx *x = (const paged_ctx *)c;
    return paged_row(x->v, x, j);
}

/*
 * Paged variant ("Shape domain" row of the Model Spec: page size 16).
 * k_pages, v_pages: [P, page_size, KVH, D] bf16 bits
 * block_table:      [B, max_pages] page ids
 * A sequence whose attended range references a page id outside [0, P) gets NaN
 * for all of its heads (the ABI's convention for a corrupt block table).
 */
int oracle_gqa_decode_paged_f64(const uint16_t *q, const uint16_t *k_pages,
                                const uint16_t *v_pages, const int32_t *block_table,
                                const int32_t *seq_lens, int B, int P, int max_pages,
                                int page_size, int H, int KVH, int D, int window,
                                int nthreads, double *out)
{
    int b;
    if (B < 0 || P <= 0 || max_pages <= 0 || page_size <= 0 || H <= 0 || KVH <= 0 || D <= 0 ||
        window < 0)
        return ORACLE_EINVAL;
    if (H % KVH != 0) return ORACLE_EINVAL;
    int64_t max_n = 1;
    for (b = 0; b < B; ++b) {
        int64_t lo, hi;
        if (seq_lens[b] < 0 || (int64_t)seq_lens[b] > (int64_t)max_pages * page_size)
            return ORACLE_EINVAL;
        attended_range(seq_lens[b], window, &lo, &hi);
        if (hi - lo > max_n) max_n = hi - lo;
    }
    const int g = H / KVH;
    const int64_t pairs = (int64_t)B * H;
    int err = ORACLE_OK;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#endif
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)max_n);
        double *q_row = (double *)malloc(sizeof(double) * (size_t)D);
        const int have_scratch = scores != NULL && q_row != NULL;
        int64_t p;
        /* every thread reaches the work-sharing loop (it ends in a barrier) */
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (p = 0; p < pairs; ++p) {
            if (!have_scratch) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                err = ORACLE_ENOMEM;
                continue;
            }
            {
                const int64_t bb = p / H, h = p % H;
                const int32_t *bt_row = block_table + bb * (int64_t)max_pages;
                double *o = out + (bb * H + h) * D;
                int64_t lo, hi, s;
                int d, bad = 0;
                attended_range(seq_lens[bb], window, &lo, &hi);
                for (s = lo; s < hi; s += 1) {
                    int32_t page = bt_row[s / page_size];
                    if (page < 0 || page >= P) {
                        bad = 1;
                        break;
                    }
                }
                if (bad) {
                    for (d = 0; d < D; ++d) o[d] = NAN;
                    continue;
                }
                for (d = 0; d < D; ++d) q_row[d] = bf16_bits_to_double(q[(bb * H + h) * D + d]);
                paged_ctx c = {k_pages, v_pages, bt_row, h / g, lo, page_size, KVH, D};
                attend(q_row, D, hi - lo, paged_k, paged_v, &c, scores, o);
            }
        }
        free(scores);
        free(q_row);
    }
    (void)nthreads;
    return err;
}

/* Threads the OpenMP runtime would use by default (for reporting). */
int oracle_default_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- window-capped (ring-buffer) cache: k, v are [B, C, KVH, D]; position s of
 *      sequence b lives at row s mod C ("Retrofit Plan: Gemma 4 31B IT ->
 *      Progressive Multi-Scale SWA with Block Attention Residuals", §3.3 and
 *      §7.3: each sliding layer keeps its own cache, capped at its window) ---- */
typedef struct {
    const uint16_t *k, *v;
    int64_t b, kvh, lo, C;
    int KVH, D;
} ring_ctx;

static const uint16_t *ring_row(const uint16_t *t, const ring_ctx *x, int64_t j)
{
    const int64_t s = x->lo + j;    /* absolute position */
    const int64_t row = s % x->C;   /* its slot in the ring */
    return t + ((x->b * x->C + row) * x->KVH + x->kvh) * x->D;
}
static const uint16_t *ring_k(const void *c, int64_t j)
{
    return ring_row(((const ring_ctx *)c)->k, (const ring_ctx *)c, j);
}
static const uint16_t *ring_v(const void *c, int64_t j)
{
    return ring_row(((const ring_ctx *)c)->v, (const ring_ctx *)c, j);
}

/*
 * Ring-buffer variant.  The attended range is the same as above, positions
 * [max(0, L_b - window), L_b); all of them are still held when 1 <= window <= C
 * (each of the last C positions has its own slot), which this function
 * requires.  L_b itself may exceed C.
 * k, v: [B, C, KVH, D] bf16 bits.
 */
int oracle_gqa_decode_ring_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                               const int32_t *seq_lens, int B, int C, int H, int KVH, int D,
                               int window, int nthreads, double *out)
{
    int b;
    if (B < 0 || C <= 0 || H <= 0 || KVH <= 0 || D <= 0 || window < 1 || window > C)
        return ORACLE_EINVAL;
    if (H % KVH != 0) return ORACLE_EINVAL;
    int64_t max_n = 1;
    for (b = 0; b < B; ++b) {
        int64_t lo, hi;
        if (seq_lens[b] < 0) return ORACLE_EINVAL;
        attended_range(seq_lens[b], window, &lo, &hi);
        if (hi - lo > max_n) max_n = hi - lo;
    }
    const int g = H / KVH;
    const int64_t pairs = (int64_t)B * H;
    int err = ORACLE_OK;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#endif
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)max_n);
        double *q_row = (double *)malloc(sizeof(double) * (size_t)D);
        const int have_scratch = scores != NULL && q_row != NULL;
        int64_t p;
        /* every thread reaches the work-sharing loop (it ends in a barrier) */
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (p = 0; p < pairs; ++p) {
            if (!have_scratch) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                err = ORACLE_ENOMEM;
                continue;
            }
            {
                const int64_t bb = p / H, h = p % H;
                int64_t lo, hi;
                int d;
                attended_range(seq_lens[bb], window, &lo, &hi);
                for (d = 0; d < D; ++d) q_row[d] = bf16_bits_to_double(q[(bb * H + h) * D + d]);
                ring_ctx c = {k, v, bb, h / g, lo, C, KVH, D};
                attend(q_row, D, hi - lo, ring_k, ring_v, &c, scores, out + (bb * H + h) * D);
            }
        }
        free(scores);
        free(q_row);
    }
    (void)nthreads;
    return err;
}

/* ---- single K=V global cache (gemma-4-31B Model Spec, "What to watch for": the
 *      global layers have values = keys; "Gemma 4 31B-it Text Architecture",
 *      decoder listing: V_raw = K_raw on full layers, K = rope(k_norm(K_raw)),
 *      V = v_norm(K_raw)).  k_norm and v_norm divide the same vector by the same
 *      root mean square, so k_norm(K_raw) = w_k * v elementwise and the key of a
 *      cached value row v at position s is
 *          k = rope(w_k * v, s)
 *      with the Model Spec's `attn.rope` row for global layers: pairs (i, i + D/2),
 *      i < n_rot, rotated by s * theta^(-2i/D):
 *          k[i]       = x[i] cos(a) - x[i + D/2] sin(a)
 *          k[i + D/2] = x[i + D/2] cos(a) + x[i] sin(a),   a = s * theta^(-2i/D)
 *      and every other coordinate unchanged (zero inverse frequency). ---- */

/* key of cached row `vr` (D bf16) at position s, in double precision */
static void derived_key(const uint16_t *vr, const double *w, int D, int n_rot, double theta,
                        int64_t s, double *k)
{
    int d, i;
    const int half = D / 2;
    for (d = 0; d < D; ++d) k[d] = w[d] * bf16_bits_to_double(vr[d]);
    for (i = 0; i < n_rot; ++i) {
        const double a = (double)s * pow(theta, -2.0 * (double)i / (double)D);
        const double c = cos(a), sn = sin(a);
        const double x0 = k[i], x1 = k[i + half];
        k[i] = x0 * c - x1 * sn;
        k[i + half] = x1 * c + x0 * sn;
    }
}

/*
 * q:        [B, H, D] bf16 bits (already normed and rotated at its own position)
 * v:        [B, S, KVH, D] bf16 bits, the cached values; row s is position s
 * w_k:      [D] bf16 bits, the layer's k_norm weight
 * n_rot, theta: rotated pairs and RoPE base (64 and 1e6 for the global layers)
 * Steps 1-5 of the definition at the top, with k derived from v as above.
 */
int oracle_gqa_decode_keqv_f64(const uint16_t *q, const uint16_t *v, const uint16_t *w_k,
                               const int32_t *seq_lens, int B, int S, int H, int KVH, int D,
                               int window, int n_rot, double theta, int nthreads, double *out)
{
    int b;
    if (B < 0 || S < 0 || H <= 0 || KVH <= 0 || D <= 0 || D % 2 != 0 || window < 0 ||
        n_rot < 0 || n_rot > D / 2 || !(theta > 0.0))
        return ORACLE_EINVAL;
    if (H % KVH != 0) return ORACLE_EINVAL;
    int64_t max_n = 1;
    for (b = 0; b < B; ++b) {
        int64_t lo, hi;
        if (seq_lens[b] < 0 || seq_lens[b] > S) return ORACLE_EINVAL;
        attended_range(seq_lens[b], window, &lo, &hi);
        if (hi - lo > max_n) max_n = hi - lo;
    }
    const int g = H / KVH;
    const int64_t pairs = (int64_t)B * H;
    int err = ORACLE_OK;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#endif
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)max_n);
        double *q_row = (double *)malloc(sizeof(double) * (size_t)D);
        double *w = (double *)malloc(sizeof(double) * (size_t)D);
        double *k = (double *)malloc(sizeof(double) * (size_t)D);
        const int have_scratch = scores && q_row && w && k;
        int64_t p;
        /* every thread reaches the work-sharing loop (it ends in a barrier) */
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (p = 0; p < pairs; ++p) {
            if (!have_scratch) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                err = ORACLE_ENOMEM;
                continue;
            }
            {
                const int64_t bb = p / H, h = p % H, kvh = h / g;
                double *o = out + (bb * H + h) * D;
                int64_t lo, hi, j;
                int d;
                attended_range(seq_lens[bb], window, &lo, &hi);
                for (d = 0; d < D; ++d) {
                    q_row[d] = bf16_bits_to_double(q[(bb * H + h) * D + d]);
                    w[d] = bf16_bits_to_double(w_k[d]);
                    o[d] = 0.0;
                }
                const int64_t n = hi - lo;
                if (n <= 0) continue; /* empty sum */
                /* 1. scores with the derived keys, scale 1 */
                for (j = 0; j < n; ++j) {
                    const int64_t s = lo + j;
                    derived_key(v + ((bb * S + s) * KVH + kvh) * D, w, D, n_rot, theta, s, k);
                    double acc = 0.0;
                    for (d = 0; d < D; ++d) acc += q_row[d] * k[d];
                    scores[j] = acc;
                }
                /* 2. max, 3. exponentials, 4. normaliser */
                double m = scores[0];
                for (j = 1; j < n; ++j)
                    if (scores[j] > m) m = scores[j];
                double l = 0.0;
                for (j = 0; j < n; ++j) {
                    scores[j] = exp(scores[j] - m);
                    l += scores[j];
                }
                /* 5. weighted sum of the cached values over the normaliser */
                for (j = 0; j < n; ++j) {
                    const uint16_t *vr = v + ((bb * S + lo + j) * KVH + kvh) * D;
                    for (d = 0; d < D; ++d) o[d] += scores[j] * bf16_bits_to_double(vr[d]);
                }
                for (d = 0; d < D; ++d) o[d] /= l;
            }
        }
        free(scores);
        free(q_row);
        free(w);
        free(k);
    }
    (void)nthreads;
    return err;
}

/* ---- decode-step producer: the nodes ahead of attn.core for one new token per
 *      sequence ("Gemma 4 31B-it Text Architecture", decoder listing: Q =
 *      rope(q_norm(Q)), K = rope(k_norm(K_raw)), V = v_norm(V_raw), with V_raw =
 *      K_raw on global layers; the new K/V are appended before attention).
 *      Model Spec rows: attn.qk_norm (per head, x / sqrt(mean x^2 + eps) * w),
 *      attn.v_norm (the same without a weight), eps 1e-6; attn.rope (pairs
 *      (i, i + D/2), i < n_rot, rotated by pos * theta^(-2i/D)).  The token's
 *      position is L - 1, L = seq_lens[b] counting the new token. ---- */

#define PRODUCER_EPS 1e-6

/* per-head RMS norm of D bf16 values; w = NULL for the unit (weightless) form */
static void rms_norm_head(const uint16_t *x, const uint16_t *w, int D, double *y)
{
    int d;
    double ss = 0.0;
    for (d = 0; d < D; ++d) {
        const double v = bf16_bits_to_double(x[d]);
        ss += v * v;
    }
    const double inv = 1.0 / sqrt(ss / (double)D + PRODUCER_EPS);
    for (d = 0; d < D; ++d) {
        y[d] = bf16_bits_to_double(x[d]) * inv;
        if (w) y[d] *= bf16_bits_to_double(w[d]);
    }
}

/* rotate the pairs (i, i + D/2), i < n_rot, by pos * theta^(-2i/D), in place */
static void rope_head(double *y, int D, int n_rot, double theta, int64_t pos)
{
    int i;
    const int half = D / 2;
    for (i = 0; i < n_rot; ++i) {
        const double a = (double)pos * pow(theta, -2.0 * (double)i / (double)D);
        const double c = cos(a), s = sin(a);
        const double x0 = y[i], x1 = y[i + half];
        y[i] = x0 * c - x1 * s;
        y[i + half] = x1 * c + x0 * s;
    }
}

/*
 * q_raw [B, H, D], k_raw [B, KVH, D], v_raw [B, KVH, D] or NULL (values = keys:
 * v = v_norm(k_raw)), w_q and w_k [D]: bf16 bits.  seq_lens [B]: lengths after the
 * append.  Outputs, in doubles: q_out [B, H, D], k_out and v_out [B, KVH, D].
 * Sequences with L < 1 have no new token: their outputs are NaN.
 */
int oracle_prepare_decode_f64(const uint16_t *q_raw, const uint16_t *k_raw, const uint16_t *v_raw,
                              const uint16_t *w_q, const uint16_t *w_k, const int32_t *seq_lens,
                              int B, int H, int KVH, int D, int n_rot, double theta,
                              double *q_out, double *k_out, double *v_out)
{
    int b, h, d;
    if (B < 0 || H <= 0 || KVH <= 0 || D <= 0 || D % 2 != 0 || n_rot < 0 || n_rot > D / 2 ||
        !(theta > 0.0))
        return ORACLE_EINVAL;
    for (b = 0; b < B; ++b) {
        const int64_t pos = (int64_t)seq_lens[b] - 1;
        for (h = 0; h < H; ++h) {
            double *y = q_out + ((int64_t)b * H + h) * D;
            if (pos < 0) {
                for (d = 0; d < D; ++d) y[d] = NAN;
                continue;
            }
            rms_norm_head(q_raw + ((int64_t)b * H + h) * D, w_q, D, y);
            rope_head(y, D, n_rot, theta, pos);
        }
        for (h = 0; h < KVH; ++h) {
            double *yk = k_out + ((int64_t)b * KVH + h) * D;
            double *yv = v_out + ((int64_t)b * KVH + h) * D;
            const uint16_t *kr = k_raw + ((int64_t)b * KVH + h) * D;
            const uint16_t *vr = v_raw ? v_raw + ((int64_t)b * KVH + h) * D : kr;
            if (pos < 0) {
                for (d = 0; d < D; ++d) yk[d] = yv[d] = NAN;
                continue;
            }
            rms_norm_head(kr, w_k, D, yk);
            rope_head(yk, D, n_rot, theta, pos);
            rms_norm_head(vr, NULL, D, yv);
        }
    }
    return ORACLE_OK;
}

/* ---- multi-query decode: T new tokens per sequence ("Gemma 4 31B-it Text
 *      Architecture", "Inference behavior: Prefill, Cache, and Long Context" and
 *      "Compact form").  The T tokens of a step are appended to the cache before
 *      attention, so with L_b the length after the append, query t (0 <= t < T)
 *      sits at position p = L_b - T + t (positions = past_seen_tokens +
 *      arange(T_current)) and sees the keys the masks allow for that position:
 *          full layers    (window == 0): s <= p          -> s in [0, p + 1)
 *          sliding layers (window  > 0): p - window < s <= p
 *                                                        -> s in [max(0, p + 1 - window), p + 1)
 *      A query whose position is negative (L_b < T - t) sees nothing and gets the
 *      empty sum, o = 0.  Tokens of the same step are causal among themselves:
 *      query t never sees the tokens after it. ---- */
static void query_range(int64_t L, int T, int t, int window, int64_t *lo, int64_t *hi)
{
    const int64_t p = L - T + t; /* position of query t */
    *hi = p + 1 > 0 ? p + 1 : 0;
    *lo = (window > 0 && *hi > window) ? *hi - window : 0;
}

/*
 * q:        [B, T, H, D] bf16 bits, query t of sequence b at position L_b - T + t
 * k, v:     [B, S, KVH, D] bf16 bits, row s = position s (the T new rows included)
 * seq_lens: [B] lengths after the append, 0 <= L_b <= S
 * out:      [B, T, H, D] doubles
 */
int oracle_gqa_decode_mq_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                             const int32_t *seq_lens, int B, int T, int S, int H, int KVH,
                             int D, int window, int nthreads, double *out)
{
    int b;
    if (B < 0 || T < 1 || S < 0 || H <= 0 || KVH <= 0 || D <= 0 || window < 0)
        return ORACLE_EINVAL;
    if (H % KVH != 0) return ORACLE_EINVAL;
    int64_t max_n = 1; /* longest attended range (scratch size) */
    for (b = 0; b < B; ++b) {
        int t;
        if (seq_lens[b] < 0 || seq_lens[b] > S) return ORACLE_EINVAL;
        for (t = 0; t < T; ++t) { /* every attended row lies in the cache */
            int64_t lo, hi;
            query_range(seq_lens[b], T, t, window, &lo, &hi);
            if (lo < 0 || hi > S) return ORACLE_EINVAL;
            if (hi - lo > max_n) max_n = hi - lo;
        }
    }
    const int g = H / KVH;
    const int64_t items = (int64_t)B * T * H;
    int err = ORACLE_OK;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#endif
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)max_n);
        double *q_row = (double *)malloc(sizeof(double) * (size_t)D);
        const int have_scratch = scores != NULL && q_row != NULL;
        int64_t it;
        /* every thread reaches the work-sharing loop (it ends in a barrier) */
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (it = 0; it < items; ++it) {
            if (!have_scratch) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                err = ORACLE_ENOMEM;
                continue;
            }
            {
                const int64_t bb = it / ((int64_t)T * H);
                const int t = (int)((it / H) % T);
                const int64_t h = it % H;
                const int64_t row = (bb * T + t) * H + h; /* [B, T, H] index */
                const int64_t kvh = h / g; /* the query head's KV head */
                int64_t lo, hi;
                int d;
                query_range(seq_lens[bb], T, t, window, &lo, &hi);
                for (d = 0; d < D; ++d) q_row[d] = bf16_bits_to_double(q[row * D + d]);
                const int64_t n = hi - lo;
                contig_ctx cq = {k, v, bb, kvh, lo, 0, S, KVH, D};
                attend(q_row, D, n, contig_k, contig_v, &cq, scores, out + row * D);
            }
        }
        free(scores);
        free(q_row);
    }
    (void)nthreads;
    return err;
}

/*
 * Paged multi-query variant: pools [P, page_size, KVH, D], block_table [B,
 * max_pages].  A query whose attended range names a page outside [0, P) gets NaN
 * for all of its heads; the other queries of the sequence are unaffected.
 */
int oracle_gqa_decode_mq_paged_f64(const uint16_t *q, const uint16_t *k_pages,
                                   const uint16_t *v_pages, const int32_t *block_table,
                                   const int32_t *seq_lens, int B, int T, int P, int max_pages,
                                   int page_size, int H, int KVH, int D, int window,
                                   int nthreads, double *out)
{
    int b;
    if (B < 0 || T < 1 || P <= 0 || max_pages <= 0 || page_size <= 0 || H <= 0 || KVH <= 0 ||
        D <= 0 || window < 0)
        return ORACLE_EINVAL;
    if (H % KVH != 0) return ORACLE_EINVAL;
    int64_t max_n = 1; /* longest attended range (scratch size) */
    for (b = 0; b < B; ++b) {
        int t;
        if (seq_lens[b] < 0 || (int64_t)seq_lens[b] > (int64_t)max_pages * page_size)
            return ORACLE_EINVAL;
        for (t = 0; t < T; ++t) { /* every attended row has a block-table entry */
            int64_t lo, hi;
            query_range(seq_lens[b], T, t, window, &lo, &hi);
            if (lo < 0 || hi > (int64_t)max_pages * page_size) return ORACLE_EINVAL;
            if (hi - lo > max_n) max_n = hi - lo;
        }
    }
    const int g = H / KVH;
    const int64_t items = (int64_t)B * T * H;
    int err = ORACLE_OK;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#endif
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)max_n);
        double *q_row = (double *)malloc(sizeof(double) * (size_t)D);
        const int have_scratch = scores != NULL && q_row != NULL;
        int64_t it;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (it = 0; it < items; ++it) {
            if (!have_scratch) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                err = ORACLE_ENOMEM;
                continue;
            }
            {
                const int64_t bb = it / ((int64_t)T * H);
                const int t = (int)((it / H) % T);
                const int64_t h = it % H;
                const int64_t row = (bb * T + t) * H + h;
                const int32_t *bt_row = block_table + bb * (int64_t)max_pages;
                double *o = out + row * D;
                const int64_t kvh = h / g;
                int64_t lo, hi, s;
                int d, bad = 0;
                query_range(seq_lens[bb], T, t, window, &lo, &hi);
                for (s = lo; s < hi; ++s) {
                    const int32_t pg = bt_row[s / page_size];
                    if (pg < 0 || pg >= P) bad = 1;
                }
                if (bad) {
                    for (d = 0; d < D; ++d) o[d] = NAN;
                    continue;
                }
                for (d = 0; d < D; ++d) q_row[d] = bf16_bits_to_double(q[row * D + d]);
                const int64_t n = hi - lo;
                paged_ctx cq = {k_pages, v_pages, bt_row, kvh, lo, page_size, KVH, D};
                attend(q_row, D, n, paged_k, paged_v, &cq, scores, o);
            }
        }
        free(scores);
        free(q_row);
    }
    (void)nthreads;
    return err;
}
