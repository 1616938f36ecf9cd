/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle for attention over a paged KV
 * cache with grouped-query heads.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the bench's CPU
 * baseline leg may load this library. It shares no code, header, table or
 * helper with the CUDA path; both sides only share the seeded input
 * generator.
 *
 * What it computes, and where each step comes from:
 *
 *  - Page translation (crucible paged attention results, paragraph on the
 *    K/V pool layout; crucible README "Layout, and why it was nearly free"):
 *    logical key position j of sequence s lives in physical page
 *    block_tables[s][j / page_size] at slot j % page_size.  Every logical
 *    page is translated on its own.
 *  - GQA head mapping (crucible results, paragraph on the GQA mapping; minfer
 *    doc 71 Excerpt A): kv_head = q_head / (Hq / Hkv).
 *  - Score (crucible results, reference kernel description): the dot of
 *    the query and key over head_dim, times `scale`.
 *  - Causal bound (crucible README "Prefill scheduling"; crucible results,
 *    paragraph on packed-row causality and future poisoning): a call carries T_s query rows for sequence s
 *    whose context (history + these rows) is L_s keys; row r sits at
 *    absolute position start + r with start = L_s - T_s and attends keys
 *    0 ..= start + r.  Decode is T_s = 1, so it attends 0 .. L_s - 1.
 *  - Sliding window (vllm.cpp PR #383 names a windowed instantiation of its
 *    decode kernel without defining it; read here the plain way): with
 *    window W > 0 a row whose causal end is e attends keys e - W + 1 ..= e
 *    (those that exist), its last W keys.  W = 0 is no window.
 *  - Softmax and weighted sum: out = sum_j w_j v_j / sum_j w_j with
 *    w_j = exp(sigma_j - max_k sigma_k).  This is the exact result the
 *    online update of the crucible results (the online-softmax experiment)
 *    reaches up to rounding order; the oracle takes it in two plain passes.
 *  - Split partial / combine (crucible README "Split-position attention";
 *    minfer doc 71 Excerpt F): a split over keys [t0, t1) is summarised by
 *    its running maximum m, its weight sum l and its unnormalised weighted
 *    sum acc; the combine rescales each split by exp(m_i - max_i m_i) and
 *    divides.  Here m is reported in base-2 units (sigma * log2 e), the
 *    convention of the library under test.
 *
 * All inputs are upcast exactly to double before any arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2 };
enum { OR_OK = 0, OR_BAD_LEN = 1, OR_BAD_PAGE = 2, OR_BAD_ARG = 3 };

typedef struct {
    int32_t num_seqs, num_q_heads, num_kv_heads, head_dim, page_size;
    int32_t num_pages, max_blocks_per_seq;
    int32_t window;              /* > 0: a row sees only its last `window` keys */
    int64_t page_stride, token_stride, head_stride; /* elements */
    double scale;
    int32_t q_dtype, kv_dtype;
    const void *q;               /* [total_q][Hq][D], row-major            */
    const int32_t *cu_q_lens;    /* [B+1]: rows of seq s are cu[s]..cu[s+1] */
    const void *k_cache;         /* addressed through the strides above    */
    const void *v_cache;
    const int32_t *block_tables; /* [B][max_blocks_per_seq]                */
    const int32_t *context_lens; /* [B]                                    */
} or_problem;

/* Deliberate-mistake switch, used only by the tests that show each pin
 * catches a plausible error.  0 = the oracle as specified. */
static int g_mutation = 0;
void or_set_mutation(int m) { g_mutation = m; }

/* ---- exact upcasts -------------------------------------------------- */

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1, e = (h >> 10) & 0x1f, f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25);    /* (1024+f) * 2^(e-25) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load(const void *base, int dtype, int64_t i)
{
    switch (dtype) {
    case OR_F32: return (double)((const float *)base)[i];
    case OR_F16: return half_bits_to_double(((const uint16_t *)base)[i]);
    default:     return bf16_bits_to_double(((const uint16_t *)base)[i]);
    }
}

double or_upcast(int dtype, const void *base, int64_t i) { return load(base, dtype, i); }

/* ---- one distribution ------------------------------------------------ */

static int seq_of_row(const or_problem *p, int64_t row)
{
    for (int s = 0; s < p->num_seqs; ++s)
        if (row < p->cu_q_lens[s + 1]) return s;
    return -1;
}

static int64_t kv_index(const or_problem *p, int32_t page, int slot, int kvh, int d)
{
    return (int64_t)page * p->page_stride + (int64_t)slot * p->token_stride +
           (int64_t)kvh * p->head_stride + d;
}

/* Attention for packed query row `row` and q head `h`.  Writes D doubles.
 * Returns OR_OK or an error code; *keys gets the number of keys attended. */
static int attend_row(const or_problem *p, int64_t row, int h, double *out,
                      double *sigma, int64_t *keys)
{
    const int D = p->head_dim, P = p->page_size;
    const int s = seq_of_row(p, row);
    if (s < 0) return OR_BAD_ARG;
    const int T = p->cu_q_lens[s + 1] - p->cu_q_lens[s];
    const int L = p->context_lens[s];
    const int r = (int)(row - p->cu_q_lens[s]);
    if (T < 1 || L < T || L > p->max_blocks_per_seq * P) return OR_BAD_LEN;

    int group = p->num_q_heads / p->num_kv_heads;
    int g = h / group;                                   /* GQA mapping */
    if (g_mutation == 1) g = h % p->num_kv_heads;        /* planted: interleaved mapping */
    const int start = L - T;
    int end = start + r;                                 /* inclusive causal end */
    if (g_mutation == 2) end = end - 1 < 0 ? 0 : end - 1; /* planted: off-by-one */
    /* sliding window: keys end - window + 1 ..= end */
    int lo = (p->window > 0 && end - p->window + 1 > 0) ? end - p->window + 1 : 0;
    if (g_mutation == 8 && lo > 0) lo -= 1;               /* planted: window one key too wide */
    const int32_t *table = p->block_tables + (int64_t)s * p->max_blocks_per_seq;
    const int64_t qbase = (row * p->num_q_heads + h) * (int64_t)D;

    double mx = -INFINITY;
    for (int j = lo; j <= end; ++j) {
        int32_t page = table[j / P];
        int slot = j % P;
        if (g_mutation == 3) slot = (j + 1) % P;          /* planted: slot shift */
        if (page < 0 || page >= p->num_pages) return OR_BAD_PAGE;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += load(p->q, p->q_dtype, qbase + d) *
                   load(p->k_cache, p->kv_dtype, kv_index(p, page, slot, g, d));
        sigma[j] = p->scale * dot;
        if (g_mutation == 4) sigma[j] = -sigma[j];       /* planted: sign flip */
        if (sigma[j] > mx) mx = sigma[j];
    }
    double den = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int j = lo; j <= end; ++j) {
        int32_t page = table[j / P];
        int slot = j % P;
        if (g_mutation == 3) slot = (j + 1) % P;
        double w = exp(sigma[j] - mx);
        if (g_mutation == 5) w = exp(sigma[j]);          /* planted: no max shift */
        den += w;
        for (int d = 0; d < D; ++d) {
            int dd = d;
            if (g_mutation == 6) dd = D - 1 - d;         /* planted: transposed V */
            out[d] += w * load(p->v_cache, p->kv_dtype, kv_index(p, page, slot, g, dd));
        }
    }
    if (g_mutation == 7) den = den + 1.0;                /* planted: wrong normaliser */
    for (int d = 0; d < D; ++d) out[d] /= den;
    *keys = (int64_t)(end - lo + 1);
    return OR_OK;
}

static int max_context(const or_problem *p)
{
    int m = 1;
    for (int s = 0; s < p->num_seqs; ++s)
        if (p->context_lens[s] > m) m = p->context_lens[s];
    return m;
}

/* Full problem: out is [total_q][Hq][D] doubles.  *keys_total (nullable)
 * receives the number of (row, head, key) terms summed.  Threads: OpenMP
 * over (row, head) when nthreads > 1. */
int or_attention(const or_problem *p, double *out, int nthreads, int64_t *keys_total)
{
    if (!p || !out || p->num_seqs < 1 || p->num_kv_heads < 1 ||
        p->num_q_heads % p->num_kv_heads != 0 || p->head_dim < 1 || p->page_size < 1)
        return OR_BAD_ARG;
    const int64_t total_q = p->cu_q_lens[p->num_seqs];
    const int64_t items = total_q * p->num_q_heads;
    const int Lmax = max_context(p);
    int err = OR_OK;
    int64_t keys = 0;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads) reduction(max : err) reduction(+ : keys)
    {
        double *sigma = (double *)malloc(sizeof(double) * (size_t)Lmax);
#pragma omp for schedule(dynamic, 4)
        for (int64_t it = 0; it < items; ++it) {
            int64_t row = it / p->num_q_heads;
            int h = (int)(it % p->num_q_heads);
            int64_t k = 0;
            int e = attend_row(p, row, h, out + it * p->head_dim, sigma, &k);
            if (e > err) err = e;
            keys += k;
        }
        free(sigma);
    }
    if (keys_total) *keys_total = keys;
    return err;
}

/* One distribution (packed row, q head) -> out[D]. */
int or_attention_one(const or_problem *p, int64_t row, int h, double *out, int64_t *keys)
{
    int64_t k = 0;
    double *sigma = (double *)malloc(sizeof(double) * (size_t)max_context(p));
    int e = attend_row(p, row, h, out, sigma, &k);
    free(sigma);
    if (keys) *keys = k;
    return e;
}

/* Split summary for decode (one query row per sequence) over keys
 * [t0, t1) of sequence s, q head h:
 *   m   = max_j sigma_j * log2(e)            (-inf when the range is empty)
 *   l   = sum_j exp(sigma_j - max sigma)
 *   acc = sum_j exp(sigma_j - max sigma) v_j
 */
int or_split_partial(const or_problem *p, int s, int h, int t0, int t1,
                     double *m_log2, double *l, double *acc)
{
    const int D = p->head_dim, P = p->page_size;
    const int g = h / (p->num_q_heads / p->num_kv_heads);
    const int L = p->context_lens[s];
    const int64_t row = p->cu_q_lens[s + 1] - 1;          /* last row of s */
    if (t1 > L) t1 = L;
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    *l = 0.0;
    *m_log2 = -INFINITY;
    if (t0 >= t1) return OR_OK;
    const int32_t *table = p->block_tables + (int64_t)s * p->max_blocks_per_seq;
    const int64_t qbase = (row * p->num_q_heads + h) * (int64_t)D;
    double *sigma = (double *)malloc(sizeof(double) * (size_t)(t1 - t0));
    double mx = -INFINITY;
    for (int j = t0; j < t1; ++j) {
        int32_t page = table[j / P];
        if (page < 0 || page >= p->num_pages) { free(sigma); return OR_BAD_PAGE; }
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += load(p->q, p->q_dtype, qbase + d) *
                   load(p->k_cache, p->kv_dtype, kv_index(p, page, j % P, g, d));
        sigma[j - t0] = p->scale * dot;
        if (sigma[j - t0] > mx) mx = sigma[j - t0];
    }
    for (int j = t0; j < t1; ++j) {
        int32_t page = table[j / P];
        double w = exp(sigma[j - t0] - mx);
        *l += w;
        for (int d = 0; d < D; ++d)
            acc[d] += w * load(p->v_cache, p->kv_dtype, kv_index(p, page, j % P, g, d));
    }
    *m_log2 = mx * 1.4426950408889634074; /* log2(e) */
    free(sigma);
    return OR_OK;
}

/* Combine n splits of one distribution: m in base-2 units.
 *   M = max_i m_i, w_i = 2^(m_i - M) (0 for m_i = -inf),
 *   out = sum_i w_i acc_i / sum_i w_i l_i   (0 when no split holds keys). */
void or_combine(int n, int D, const double *m_log2, const double *l,
                const double *acc, double *out)
{
    double M = -INFINITY;
    for (int i = 0; i < n; ++i)
        if (m_log2[i] > M) M = m_log2[i];
    double den = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (M == -INFINITY) return;
    for (int i = 0; i < n; ++i) {
        if (m_log2[i] == -INFINITY) continue;
        double w = exp2(m_log2[i] - M);
        den += w * l[i];
        for (int d = 0; d < D; ++d) out[d] += w * acc[(int64_t)i * D + d];
    }
    for (int d = 0; d < D; ++d) out[d] = den > 0.0 ? out[d] / den : 0.0;
}

int or_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
