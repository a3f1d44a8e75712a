/*
 * attn_oracle.c -- plain fp64 CPU attention, materialised one query row at a time.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links or calls this
 * file; the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg use it to decide whether the GPU kernel is right.  It shares no code,
 * header or constant with the CUDA library.
 *
 * What it computes (the dense path of the aiml.sh page "Speed up long contexts
 * with FlashAttention", lab.py, `standard_attention`, generalised to an
 * explicit scale and to a non-causal mask):
 *
 *   for a query row i of head bh, with keys J_i = {0..i} (causal) or {0..N-1}:
 *     s_j  = scale * sum_c q[i][c] * k[j][c]          (j in J_i)
 *     m    = max_j s_j                                 (the page's subtract_max)
 *     e_j  = exp(s_j - m);   l = sum_j e_j
 *     p_j  = e_j / l                                   (materialised probabilities)
 *     o[c] = sum_j p_j * v[j][c]
 *     lse  = m + log(l)   -- natural-log logsumexp of the scaled, masked scores;
 *                            the pages never compute it, this is its plain definition.
 *
 * Everything is double precision, summed in index order, compiled without
 * floating-point contraction so x86 and Arm hosts produce the same bits.
 * Inputs are either doubles or bf16 bit patterns (widened exactly to double).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORACLE_IN_F64 = 0, ORACLE_IN_BF16 = 1 };

static double widen_bf16(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const void *q, *k, *v;
    int kind;
    int64_t BH, N, d;
    const int64_t *rows; /* nrows pairs (bh, i) */
    int64_t nrows;
    int causal;
    double scale;
    double *o, *lse;
    int64_t next; /* shared work cursor, advanced atomically */
    int64_t chunk;
    int failed;
} oracle_job;

static void copy_row(const void *m, int kind, int64_t N, int64_t d, int64_t bh, int64_t r,
                     double *dst)
{
    int64_t off = (bh * N + r) * d;
    if (kind == ORACLE_IN_BF16) {
        const uint16_t *p = (const uint16_t *)m + off;
        for (int64_t c = 0; c < d; ++c)
            dst[c] = widen_bf16(p[c]);
    } else {
        memcpy(dst, (const double *)m + off, (size_t)d * sizeof(double));
    }
}

static void *oracle_worker(void *arg)
{
    oracle_job *job = (oracle_job *)arg;
    const int64_t N = job->N, d = job->d;
    /* per-thread copy of the current head's K and V rows, widened to double */
    double *kc = (double *)malloc((size_t)(N * d) * sizeof(double));
    double *vc = (double *)malloc((size_t)(N * d) * sizeof(double));
    double *e = (double *)malloc((size_t)N * sizeof(double));
    double *qi = (double *)malloc((size_t)d * sizeof(double));
    double *acc = (double *)malloc((size_t)d * sizeof(double));
    if (!kc || !vc || !e || !qi || !acc) {
        __atomic_store_n(&job->failed, 1, __ATOMIC_RELAXED);
        free(kc); free(vc); free(e); free(qi); free(acc);
        return NULL;
    }
    int64_t cached_bh = -1, cached_rows = 0;

    for (;;) {
        int64_t start = __atomic_fetch_add(&job->next, job->chunk, __ATOMIC_RELAXED);
        if (start >= job->nrows)
            break;
        int64_t stop = start + job->chunk < job->nrows ? start + job->chunk : job->nrows;
        for (int64_t r = start; r < stop; ++r) {
            const int64_t bh = job->rows[2 * r], i = job->rows[2 * r + 1];
            const int64_t nkeys = job->causal ? i + 1 : N;
            if (bh != cached_bh) {
                cached_bh = bh;
                cached_rows = 0;
            }
            for (; cached_rows < nkeys; ++cached_rows) {
                copy_row(job->k, job->kind, N, d, bh, cached_rows, kc + cached_rows * d);
                copy_row(job->v, job->kind, N, d, bh, cached_rows, vc + cached_rows * d);
            }
            copy_row(job->q, job->kind, N, d, bh, i, qi);

            /* scores and their maximum */
            double m = -INFINITY;
            for (int64_t j = 0; j < nkeys; ++j) {
                const double *kj = kc + j * d;
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c)
                    dot += qi[c] * kj[c];
                e[j] = dot * job->scale;
                if (e[j] > m)
                    m = e[j];
            }
            /* exponentials shifted by the maximum, their sum, then probabilities */
            double l = 0.0;
            for (int64_t j = 0; j < nkeys; ++j) {
                e[j] = exp(e[j] - m);
                l += e[j];
            }
            for (int64_t j = 0; j < nkeys; ++j)
                e[j] = e[j] / l;
            /* probability-weighted sum of value rows */
            for (int64_t c = 0; c < d; ++c)
                acc[c] = 0.0;
            for (int64_t j = 0; j < nkeys; ++j) {
                const double pj = e[j];
                const double *vj = vc + j * d;
                for (int64_t c = 0; c < d; ++c)
                    acc[c] += pj * vj[c];
            }
            memcpy(job->o + r * d, acc, (size_t)d * sizeof(double));
            if (job->lse)
                job->lse[r] = m + log(l);
        }
    }
    free(kc); free(vc); free(e); free(qi); free(acc);
    return NULL;
}

/*
 * oracle_attn_rows: attention output and logsumexp for a list of query rows.
 *
 *   q, k, v  [BH, N, d] row-major, doubles (kind 0) or bf16 bit patterns (kind 1)
 *   rows     nrows pairs (bh, i), grouped by bh for cache reuse (any order is correct)
 *   o        out: nrows x d doubles;  lse: out, nrows doubles (may be NULL)
 *   nthreads 0 = one per online CPU
 * Returns 0 on success, -1 on a bad argument or row index, -2 if memory ran out.
 */
int oracle_attn_rows(const void *q, const void *k, const void *v, int kind, int64_t BH,
                     int64_t N, int64_t d, const int64_t *rows, int64_t nrows, int causal,
                     double scale, double *o, double *lse, int nthreads)
{
    if (!q || !k || !v || !o || (nrows > 0 && !rows) || BH < 0 || N < 0 || d <= 0 || nrows < 0)
        return -1;
    if (kind != ORACLE_IN_F64 && kind != ORACLE_IN_BF16)
        return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[2 * r] < 0 || rows[2 * r] >= BH || rows[2 * r + 1] < 0 || rows[2 * r + 1] >= N)
            return -1;
    if (nrows == 0)
        return 0;
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    if (nthreads > nrows)
        nthreads = (int)nrows;
    if (nthreads > 512)
        nthreads = 512;

    oracle_job job = {q, k, v, kind, BH, N, d, rows, nrows, causal, scale, o, lse, 0, 0, 0};
    job.chunk = nrows / ((int64_t)nthreads * 8);
    if (job.chunk < 1)
        job.chunk = 1;
    if (job.chunk > 64)
        job.chunk = 64;

    pthread_t tid[512];
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[started], NULL, oracle_worker, &job) != 0)
            break;
        ++started;
    }
    oracle_worker(&job);
    for (int t = 0; t < started; ++t)
        pthread_join(tid[t], NULL);
    return job.failed ? -2 : 0;
}

/* number of worker threads a call with nthreads = 0 would use */
int oracle_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}
