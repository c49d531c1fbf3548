/*
 * pkv_oracle.c -- plain, slow fp64 CPU oracle for single-token grouped-query
 * decode attention over a block-table paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the CPU
 * baseline leg of the benchmark are the only callers.  Nothing here is shared
 * with the CUDA path (no headers, no helpers, no tables), and the product
 * library never loads this file.
 *
 * What is computed follows "PersistentKV: Page-Aware Decode Scheduling for
 * Long-Context LLM Serving on Commodity GPUs" (gist.science summary),
 * Technical Summary / Methodology section 1 "Native Block-Table Decode Engine":
 *   - G = Hq / Hkv query heads share one KV head (grouped-query attention);
 *   - K and V live in fixed-size pages reached through a per-sequence block
 *     table and are never repacked ("Layout");
 *   - the sequence may be cut into disjoint ranges whose partial softmax states
 *     a merge step combines exactly ("Sequence Splitting").
 * The pages never write out the attention formula itself.  The reading taken
 * here is standard scaled dot-product attention of one new query token:
 *     kvh    = floor(h / G)
 *     s_t    = (1/sqrt(D)) * sum_d q[b][h][d] * K_t[kvh][d]     for t < N_b
 *     m      = max_t s_t,  l = sum_t exp(s_t - m)
 *     out    = sum_t exp(s_t - m) * V_t[kvh] / l
 *     lse    = m + ln(l)                                (natural logarithm)
 * with token t of row b at page block_table[b][t / ps], slot t % ps.
 * An empty token range gives the neutral state out = 0, lse = -inf
 * (Methodology section 1 "Row-Local Bounds": empty splits write neutral states).
 *
 * Arithmetic is fp64 on the exactly decoded bf16 inputs.  Every loop runs in
 * the plain order of the definition; there is no blocking, fusion or online
 * rescaling.
 *
 * Memory layouts (all row-major, all caller-owned):
 *   q            uint16 bf16 bits  [B][Hq][D]
 *   k_pages      uint16 bf16 bits  [num_pages][page_size][Hkv][D]
 *   v_pages      same as k_pages
 *   block_table  int32             [B][max_pages]
 *   seq_lens     int32             [B]
 *   out          double            [B][Hq][D]
 *   lse          double            [B][Hq]
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ENOMEM -2

typedef struct {
    const uint16_t *q, *k_pages, *v_pages;
    const int32_t *block_table, *seq_lens;
    int B, Hq, Hkv, D, page_size, max_pages, num_pages;
} oracle_problem;

/* bf16 is the top half of an IEEE binary32; widening is exact. */
static double bf16_value(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Address of token t of row b for KV head kvh inside a page pool. */
static const uint16_t *token_row(const oracle_problem *p, const uint16_t *pool,
                                 int b, int t, int kvh) {
    int32_t page = p->block_table[(size_t)b * p->max_pages + t / p->page_size];
    int slot = t % p->page_size;
    size_t index = (((size_t)page * p->page_size + slot) * p->Hkv + kvh) * p->D;
    return pool + index;
}

static int check_problem(const oracle_problem *p) {
    if (p->B < 0 || p->Hq <= 0 || p->Hkv <= 0 || p->D <= 0 || p->page_size <= 0 ||
        p->max_pages < 0 || p->num_pages < 0)
        return ORACLE_EINVAL;
    if (p->Hq % p->Hkv != 0) return ORACLE_EINVAL;
    for (int b = 0; b < p->B; ++b) {
        int n = p->seq_lens[b];
        if (n < 0 || n > p->max_pages * p->page_size) return ORACLE_EINVAL;
        int pages = (n + p->page_size - 1) / p->page_size;
        for (int i = 0; i < pages; ++i) {
            int32_t page = p->block_table[(size_t)b * p->max_pages + i];
            if (page < 0 || page >= p->num_pages) return ORACLE_EINVAL;
        }
    }
    return ORACLE_OK;
}

/*
 * Attention of query head h of row b over tokens [t_begin, t_end) only.
 * With the full range this is the definition above; with a sub-range it is the
 * partial softmax state of one split (normalised output and its log-sum-exp).
 * `scores` is caller scratch of at least t_end - t_begin doubles.
 */
static void attend_range(const oracle_problem *p, int b, int h, int t_begin,
                         int t_end, double *scores, double *out, double *lse) {
    const int D = p->D;
    const int G = p->Hq / p->Hkv;
    const int kvh = h / G;
    const double scale = 1.0 / sqrt((double)D);
    const uint16_t *qrow = p->q + ((size_t)b * p->Hq + h) * D;

    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (t_end <= t_begin) {
        *lse = -INFINITY;
        return;
    }

    /* s_t = scale * <q, k_t> */
    for (int t = t_begin; t < t_end; ++t) {
        const uint16_t *krow = token_row(p, p->k_pages, b, t, kvh);
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += bf16_value(qrow[d]) * bf16_value(krow[d]);
        scores[t - t_begin] = scale * dot;
    }

    /* m = max s_t */
    double m = scores[0];
    for (int t = t_begin + 1; t < t_end; ++t)
        if (scores[t - t_begin] > m) m = scores[t - t_begin];

    /* l = sum exp(s_t - m);  acc = sum exp(s_t - m) v_t */
    double l = 0.0;
    for (int t = t_begin; t < t_end; ++t) {
        double w = exp(scores[t - t_begin] - m);
        const uint16_t *vrow = token_row(p, p->v_pages, b, t, kvh);
        l += w;
        for (int d = 0; d < D; ++d) out[d] += w * bf16_value(vrow[d]);
    }

    for (int d = 0; d < D; ++d) out[d] /= l;
    *lse = m + log(l);
}

typedef struct {
    const oracle_problem *p;
    double *out, *lse;
    int unit_begin, unit_end; /* units are (b, h) pairs, h fastest */
    int status;
} oracle_job;

static void *run_units(void *arg) {
    oracle_job *job = (oracle_job *)arg;
    const oracle_problem *p = job->p;
    int longest = 0;
    for (int b = 0; b < p->B; ++b)
        if (p->seq_lens[b] > longest) longest = p->seq_lens[b];
    double *scores = (double *)malloc(sizeof(double) * (size_t)(longest > 0 ? longest : 1));
    if (!scores) {
        job->status = ORACLE_ENOMEM;
        return NULL;
    }
    for (int u = job->unit_begin; u < job->unit_end; ++u) {
        int b = u / p->Hq, h = u % p->Hq;
        attend_range(p, b, h, 0, p->seq_lens[b], scores,
                     job->out + ((size_t)b * p->Hq + h) * p->D,
                     job->lse + (size_t)b * p->Hq + h);
    }
    free(scores);
    job->status = ORACLE_OK;
    return NULL;
}

/*
 * Full decode attention for every (row, query head).  `nthreads` > 1 hands
 * disjoint (row, head) ranges to POSIX threads; each unit is computed exactly as
 * in the single-threaded case, so the result does not depend on nthreads.
 */
int pkv_oracle_decode(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                      const int32_t *block_table, const int32_t *seq_lens, int B, int Hq,
                      int Hkv, int D, int page_size, int max_pages, int num_pages,
                      double *out, double *lse, int nthreads) {
    oracle_problem p = {q, k_pages, v_pages, block_table, seq_lens,
                        B, Hq, Hkv, D, page_size, max_pages, num_pages};
    int rc = check_problem(&p);
    if (rc != ORACLE_OK) return rc;
    int units = B * Hq;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > units) nthreads = units > 0 ? units : 1;

    oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t *threads = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !threads) {
        free(jobs);
        free(threads);
        return ORACLE_ENOMEM;
    }
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].p = &p;
        jobs[i].out = out;
        jobs[i].lse = lse;
        jobs[i].unit_begin = (int)((long long)units * i / nthreads);
        jobs[i].unit_end = (int)((long long)units * (i + 1) / nthreads);
    }
    if (nthreads == 1) {
        run_units(&jobs[0]);
    } else {
        for (int i = 0; i < nthreads; ++i) pthread_create(&threads[i], NULL, run_units, &jobs[i]);
        for (int i = 0; i < nthreads; ++i) pthread_join(threads[i], NULL);
    }
    rc = ORACLE_OK;
    for (int i = 0; i < nthreads; ++i)
        if (jobs[i].status != ORACLE_OK) rc = jobs[i].status;
    free(jobs);
    free(threads);
    return rc;
}

/*
 * Partial state of one split: the G query heads of KV head `kvh` in row b,
 * attending only to tokens [token_begin, min(token_end, N_b)).
 * out is [G][D] (normalised within the split), lse is [G].
 */
int pkv_oracle_partial(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                       const int32_t *block_table, const int32_t *seq_lens, int B, int Hq,
                       int Hkv, int D, int page_size, int max_pages, int num_pages, int b,
                       int kvh, int token_begin, int token_end, double *out, double *lse) {
    oracle_problem p = {q, k_pages, v_pages, block_table, seq_lens,
                        B, Hq, Hkv, D, page_size, max_pages, num_pages};
    int rc = check_problem(&p);
    if (rc != ORACLE_OK) return rc;
    if (b < 0 || b >= B || kvh < 0 || kvh >= Hkv || token_begin < 0) return ORACLE_EINVAL;
    int n = seq_lens[b];
    if (token_end > n) token_end = n;
    int G = Hq / Hkv;
    int len = token_end > token_begin ? token_end - token_begin : 1;
    double *scores = (double *)malloc(sizeof(double) * (size_t)len);
    if (!scores) return ORACLE_ENOMEM;
    for (int g = 0; g < G; ++g)
        attend_range(&p, b, kvh * G + g, token_begin, token_end, scores,
                     out + (size_t)g * D, lse + g);
    free(scores);
    return ORACLE_OK;
}

/*
 * Exact merge of S partial states of one query head (Methodology section 1,
 * "A separate merge kernel combines these states exactly").  With
 * M = max_s lse_s and w_s = exp(lse_s - M):
 *     out = sum_s w_s * o_s / sum_s w_s,      lse = M + ln(sum_s w_s).
 * A neutral part (lse_s = -inf) has weight 0; if every part is neutral the
 * result is the neutral state.
 * o_parts is [S][D], lse_parts is [S].
 */
void pkv_oracle_merge(const double *o_parts, const double *lse_parts, int S, int D,
                      double *out, double *lse) {
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    double M = -INFINITY;
    for (int s = 0; s < S; ++s)
        if (lse_parts[s] > M) M = lse_parts[s];
    if (M == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double wsum = 0.0;
    for (int s = 0; s < S; ++s) {
        if (lse_parts[s] == -INFINITY) continue;
        double w = exp(lse_parts[s] - M);
        wsum += w;
        for (int d = 0; d < D; ++d) out[d] += w * o_parts[(size_t)s * D + d];
    }
    for (int d = 0; d < D; ++d) out[d] /= wsum;
    *lse = M + log(wsum);
}
