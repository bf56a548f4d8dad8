/*
 * FP64 CPU oracle for paged attention with asymmetric K/V head dims.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may build, load or call this file. The GPU
 * library never links it and it shares no code, header, table or helper with
 * the GPU library.
 *
 * What it computes (plain definition, no blocking, no reordering):
 *   For request b, query token t in [0, n_b), query head h:
 *     g  = h / (Hq / Hkv)                       consecutive q heads share a KV head
 *     i  = L_b - n_b + t                        the new tokens are the last n_b keys
 *     V  = { j : 0 <= j <= i and (W <= 0 or j > i - W) }
 *     k_j = dec(K[page_table[b][j / P], j % P, g, :]) * k_scale
 *     v_j = dec(V[page_table[b][j / P], j % P, g, :]) * v_scale
 *     s_j = softmax_scale * <q, k_j>
 *     m   = max(max_j s_j, sigma_h)             sigma_h = -inf without sinks
 *     Z   = sum_j exp(s_j - m) + exp(sigma_h - m)
 *     out = sum_j exp(s_j - m) v_j / Z ,  lse = m + ln Z
 *
 * Sources (the pages give no formula; these are the readings, listed in the
 * design notes):
 *   - head dims QK=192 / V=128 carried separately: sglang PR #32818
 *     ("Route asymmetric-KV models to fa4", change 1 and the trtllm_mha check);
 *   - paged KV, page size 1 or 128: sglang PR #41886, "Speed Tests";
 *   - decode, 8-token verify, full vs SWA with sinks, ragged page boundaries:
 *     sglang PR #41886, "Accuracy Tests";
 *   - unused KV tails may hold NaN and must be masked, not multiplied:
 *     sammysun0711/sglang PR #35, "Modifications" (FlyPA V-tail masking) and
 *     its test list (test_mimo_flypa_nan_tail.py);
 *   - verify as one causal block per request, split-KV with a merge:
 *     MiMo-V2.6-Flash-RL model card, "What the kernels do";
 *   - FP8 E4M3 K/V converted to a wide type before Q.K (Q stays wide; FP8
 *     Q.K was measured and rejected): same model card, "What the kernels do"
 *     and "Things that were measured and did not help".
 *
 * Every visible key is read; no other slot is ever read, so the contents of
 * unused slots (NaN included) cannot reach the result.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ORACLE_MUTANT selects a deliberately wrong variant (0 = the oracle itself).
 * The pin tests build each mutant and require that some pin rejects it; this
 * shows that a plausible slip in any step would not go unnoticed. */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* Exact widening of a bfloat16 bit pattern: the bf16 bits are the top half
 * of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Exact widening of an OCP FP8 E4M3 ("e4m3fn") code, from the format
 * definition: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent field 0 encodes subnormals m/8 * 2^-6; S.1111.111 is NaN; there
 * is no infinity. */
double oracle_e4m3_to_double(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - (ORACLE_MUTANT == 8 ? 8 : 7));
    return sign ? -mag : mag;
}

typedef struct {
    int batch, hq, hkv, dqk, dv;
    int page_size, page_table_stride, kv_dtype; /* 0 = bf16, 1 = e4m3 */
    int window;
    int64_t num_pages;
    double softmax_scale, k_scale, v_scale;
    const int32_t *qo_indptr, *seq_lens, *page_table;
    const uint16_t *q;
    const void *k_cache, *v_cache;
    const double *sinks; /* [hq] or NULL */
} oracle_problem_t;

static double kv_elem(const oracle_problem_t *p, const void *cache, int64_t idx)
{
    if (p->kv_dtype == 0)
        return oracle_bf16_to_double(((const uint16_t *)cache)[idx]);
    return oracle_e4m3_to_double(((const uint8_t *)cache)[idx]);
}

/* Physical slot of logical key j of request b, or -1 if the page id is out of
 * the pool. */
static int64_t slot_of(const oracle_problem_t *p, int b, int64_t j)
{
    int64_t page = p->page_table[(int64_t)b * p->page_table_stride + j / p->page_size];
    if (page < 0 || page >= p->num_pages)
        return -1;
    int64_t off = j % p->page_size;
    if (ORACLE_MUTANT == 5)
        off = p->page_size - 1 - off;
    return page * p->page_size + off;
}

/* Request b that owns flat query token `tok` (qo_indptr is monotone). */
static int request_of(const oracle_problem_t *p, int64_t tok)
{
    int b = 0;
    while (b + 1 < p->batch && p->qo_indptr[b + 1] <= tok)
        b++;
    return b;
}

/*
 * One output row (query token `tok`, head h) restricted to logical keys in
 * [key_lo, key_hi) intersected with the visible set.
 *   with_sink = 1: out = sum_j e^{s_j-m} v_j / Z with the sink term in Z, and
 *                  lse = m + ln Z (the full definition above when the range
 *                  covers every key);
 *   with_sink = 0: the same without the sink term (a split partial).
 * An empty visible range with no sink gives out = 0 and lse = -inf.
 * `scores` is scratch of at least key_hi - key_lo doubles.
 * Returns 0, or -1 when a visible key maps outside the pool.
 */
static int one_row(const oracle_problem_t *p, int64_t tok, int h, int64_t key_lo,
                   int64_t key_hi, int with_sink, double *scores, double *out,
                   double *lse)
{
    const int b = request_of(p, tok);
    const int64_t n_b = p->qo_indptr[b + 1] - p->qo_indptr[b];
    const int64_t L = p->seq_lens[b];
    const int64_t t = tok - p->qo_indptr[b];
    const int64_t i = (ORACLE_MUTANT == 4) ? t : L - n_b + t;
    const int G = p->hq / p->hkv;
    const int g = (ORACLE_MUTANT == 2) ? h % p->hkv : h / G;
    const int gv = (ORACLE_MUTANT == 10) ? (g + 1) % p->hkv : g;
    const uint16_t *qrow = p->q + (tok * p->hq + h) * (int64_t)p->dqk;

    /* visible set: j <= i, and j > i - W when a window is set */
    int64_t lo = 0, hi = i + 1;
    const int64_t wlo = (ORACLE_MUTANT == 3) ? i - p->window : i - p->window + 1;
    if (p->window > 0 && wlo > lo)
        lo = wlo;
    if (key_lo > lo)
        lo = key_lo;
    if (key_hi < hi)
        hi = key_hi;

    double sink = -INFINITY;
    if (with_sink && p->sinks)
        sink = p->sinks[h];

    double m = sink;
    for (int64_t j = lo; j < hi; j++) {
        int64_t slot = slot_of(p, b, j);
        if (slot < 0)
            return -1;
        const int64_t base = (slot * p->hkv + g) * (int64_t)p->dqk;
        const double ks = (ORACLE_MUTANT == 6) ? 1.0 : p->k_scale;
        const int dmax = (ORACLE_MUTANT == 9) ? p->dqk - 1 : p->dqk;
        double dot = 0.0;
        for (int d = 0; d < dmax; d++)
            dot += oracle_bf16_to_double(qrow[d]) * (kv_elem(p, p->k_cache, base + d) * ks);
        double s = p->softmax_scale * dot;
        scores[j - lo] = s;
        if (s > m)
            m = s;
    }

    for (int d = 0; d < p->dv; d++)
        out[d] = 0.0;
    if (m == -INFINITY) { /* nothing visible and no sink */
        *lse = -INFINITY;
        return 0;
    }

    double Z = (ORACLE_MUTANT == 1) ? 0.0 : exp(sink - m);
    const double vs = (ORACLE_MUTANT == 7) ? 1.0 : p->v_scale;
    for (int64_t j = lo; j < hi; j++) {
        double w = exp(scores[j - lo] - m);
        Z += w;
        const int64_t base = (slot_of(p, b, j) * p->hkv + gv) * (int64_t)p->dv;
        for (int d = 0; d < p->dv; d++)
            out[d] += w * (kv_elem(p, p->v_cache, base + d) * vs);
    }
    for (int d = 0; d < p->dv; d++)
        out[d] /= Z;
    *lse = (ORACLE_MUTANT == 11) ? m : m + log(Z);
    return 0;
}

static int64_t max_seq_len(const oracle_problem_t *p)
{
    int64_t mx = 1;
    for (int b = 0; b < p->batch; b++)
        if (p->seq_lens[b] > mx)
            mx = p->seq_lens[b];
    return mx;
}

/*
 * Rows to compute: rows[r] = tok * Hq + h (NULL: every row in order).
 * out: [n_rows, dv] doubles, lse: [n_rows] doubles (may be NULL).
 * key_lo/key_hi restrict the keys (pass 0 / INT64_MAX for all);
 * with_sink selects the full row (1) or a split partial (0).
 * Returns 0, or -1 if any visible key maps outside the pool.
 */
static int run_rows(const oracle_problem_t *p, const int64_t *rows, int64_t n_rows,
                    int64_t key_lo, int64_t key_hi, int with_sink, double *out,
                    double *lse, int nthreads)
{
    const int64_t scratch = max_seq_len(p);
    int status = 0;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)scratch);
        if (!scores) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = -2;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t r = 0; r < n_rows; r++) {
                int64_t row = rows ? rows[r] : r;
                double l;
                int rc = one_row(p, row / p->hq, (int)(row % p->hq), key_lo, key_hi,
                                 with_sink, scores, out + r * (int64_t)p->dv, &l);
                if (lse)
                    lse[r] = l;
                if (rc) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                    status = rc;
                }
            }
            free(scores);
        }
    }
    (void)nthreads;
    return status;
}

#define ORACLE_PROBLEM_ARGS                                                             \
    int batch, int hq, int hkv, int dqk, int dv, int page_size, int page_table_stride,  \
        int kv_dtype, int window, int64_t num_pages, double softmax_scale,              \
        double k_scale, double v_scale, const int32_t *qo_indptr,                       \
        const int32_t *seq_lens, const int32_t *page_table, const uint16_t *q,          \
        const void *k_cache, const void *v_cache, const double *sinks

static oracle_problem_t make_problem(ORACLE_PROBLEM_ARGS)
{
    oracle_problem_t p;
    p.batch = batch; p.hq = hq; p.hkv = hkv; p.dqk = dqk; p.dv = dv;
    p.page_size = page_size; p.page_table_stride = page_table_stride;
    p.kv_dtype = kv_dtype; p.window = window; p.num_pages = num_pages;
    p.softmax_scale = softmax_scale; p.k_scale = k_scale; p.v_scale = v_scale;
    p.qo_indptr = qo_indptr; p.seq_lens = seq_lens; p.page_table = page_table;
    p.q = q; p.k_cache = k_cache; p.v_cache = v_cache; p.sinks = sinks;
    return p;
}

static int check_problem(const oracle_problem_t *p)
{
    if (p->batch < 0 || p->hq <= 0 || p->hkv <= 0 || p->hq % p->hkv || p->page_size <= 0)
        return -3;
    for (int b = 0; b < p->batch; b++) {
        int64_t n = (int64_t)p->qo_indptr[b + 1] - p->qo_indptr[b];
        if (n < 0 || p->seq_lens[b] < n)
            return -3;
        if ((p->seq_lens[b] + p->page_size - 1) / p->page_size > p->page_table_stride)
            return -3;
    }
    return 0;
}

/* The attention rows listed in `rows` (or all rows) with the sink term. */
int oracle_attn_paged(ORACLE_PROBLEM_ARGS, const int64_t *rows, int64_t n_rows,
                      double *out, double *lse, int nthreads)
{
    oracle_problem_t p = make_problem(batch, hq, hkv, dqk, dv, page_size, page_table_stride,
                                      kv_dtype, window, num_pages, softmax_scale, k_scale,
                                      v_scale, qo_indptr, seq_lens, page_table, q, k_cache,
                                      v_cache, sinks);
    int rc = check_problem(&p);
    if (rc)
        return rc;
    if (!rows)
        n_rows = (int64_t)qo_indptr[batch] * hq;
    return run_rows(&p, rows, n_rows, 0, INT64_MAX, 1, out, lse, nthreads);
}

/* A split partial: keys restricted to [key_lo, key_hi), no sink, output
 * normalised by its own denominator, lse = m + ln(sum e^{s-m}) (-inf when
 * the range holds no visible key). */
int oracle_attn_partial(ORACLE_PROBLEM_ARGS, int64_t key_lo, int64_t key_hi,
                        const int64_t *rows, int64_t n_rows, double *out, double *lse,
                        int nthreads)
{
    oracle_problem_t p = make_problem(batch, hq, hkv, dqk, dv, page_size, page_table_stride,
                                      kv_dtype, window, num_pages, softmax_scale, k_scale,
                                      v_scale, qo_indptr, seq_lens, page_table, q, k_cache,
                                      v_cache, sinks);
    int rc = check_problem(&p);
    if (rc)
        return rc;
    if (!rows)
        n_rows = (int64_t)qo_indptr[batch] * hq;
    return run_rows(&p, rows, n_rows, key_lo, key_hi, 0, out, lse, nthreads);
}

/*
 * Log-sum-exp combine of S split partials of one row (the merge that a
 * split-KV schedule needs; the model card names split-KV, the combine rule is
 * the standard one):
 *   M = max(max_s lse_s, sigma);  w_s = e^{lse_s - M};
 *   Z = sum_s w_s + e^{sigma - M};  out = sum_s w_s o_s / Z;  lse = M + ln Z.
 * Partials with lse = -inf carry no weight (their o_s is not read).
 * o_parts: [S, dv]; sigma = -inf for no sink.
 */
void oracle_merge(int num_splits, int dv, const double *o_parts, const double *lse_parts,
                  double sigma, double *out, double *lse)
{
    double M = sigma;
    for (int s = 0; s < num_splits; s++)
        if (lse_parts[s] > M)
            M = lse_parts[s];
    for (int d = 0; d < dv; d++)
        out[d] = 0.0;
    if (M == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double Z = exp(sigma - M);
    for (int s = 0; s < num_splits; s++) {
        if (lse_parts[s] == -INFINITY)
            continue;
        double w = exp(lse_parts[s] - M);
        Z += w;
        for (int d = 0; d < dv; d++)
            out[d] += w * o_parts[(int64_t)s * dv + d];
    }
    for (int d = 0; d < dv; d++)
        out[d] /= Z;
    *lse = M + log(Z);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
