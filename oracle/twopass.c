/* O2 — streaming two-pass attention forward in plain C, fp64.
 * TEST INFRASTRUCTURE ONLY: called from the tests and from bench.py's CPU
 * baseline through ctypes; the GPU library never links it.
 *
 * The definition is softmax(scale * Q K^T [masked]) V with a per-row natural
 * log-sum-exp, as in wiki.ai-engineering.at "Flash Attention" ("Das
 * Grundproblem") and johe.ru "Flash Attention: ..." ("Введение").  This file
 * computes it without materialising the score matrix, one query row at a
 * time, in the classical "safe softmax" order, streaming the keys in blocks:
 *
 *   pass 1a: M_i = max_j s_ij                   (s_ij = scale * q_i . k_j)
 *   pass 1b: l_i = sum_j exp(s_ij - M_i)
 *   pass 2 : O_i = sum_j exp(s_ij - M_i) / l_i * v_j,  LSE_i = M_i + log l_i
 *
 * Scores are recomputed in every pass (nothing of size Nk is stored).  Masking
 * is bottom-right causal (key j visible to query i iff j <= i + Nk - Nq); a row
 * with no visible key gets O = 0 and LSE = -inf.  Rows are shared among
 * `nthreads` POSIX threads.  Inputs are fp64 arrays [BH, N, d] contiguous.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

typedef struct {
    const double *q, *k, *v;
    double *o, *lse;
    int64_t BH, Nq, Nk, d, dv;
    double scale;
    int causal;
    int64_t block;
    const int64_t *rows; /* optional: query index of each of the R given rows */
    int64_t R;           /* rows per head given in q / written to o, lse */
    int64_t row_begin, row_end; /* flattened (bh, r) rows */
} job_t;

static double dot(const double *a, const double *b, int64_t n) {
    double s = 0.0;
    for (int64_t c = 0; c < n; ++c) s += a[c] * b[c];
    return s;
}

static void one_row(const job_t *J, int64_t bh, int64_t r) {
    int64_t i = J->rows ? J->rows[r] : r; /* query index, for the causal limit */
    const double *qi = J->q + (bh * J->R + r) * J->d;
    const double *K = J->k + bh * J->Nk * J->d;
    const double *V = J->v + bh * J->Nk * J->dv;
    double *oi = J->o + (bh * J->R + r) * J->dv;
    int64_t nvis = J->Nk;
    if (J->causal) {
        int64_t lim = i + J->Nk - J->Nq; /* last visible key */
        nvis = lim + 1 < 0 ? 0 : (lim + 1 > J->Nk ? J->Nk : lim + 1);
    }
    for (int64_t c = 0; c < J->dv; ++c) oi[c] = 0.0;
    if (nvis == 0) {
        J->lse[bh * J->R + r] = -INFINITY;
        return;
    }
    /* pass 1a: row maximum, streamed over key blocks */
    double M = -INFINITY;
    for (int64_t j0 = 0; j0 < nvis; j0 += J->block) {
        int64_t j1 = j0 + J->block < nvis ? j0 + J->block : nvis;
        for (int64_t j = j0; j < j1; ++j) {
            double s = J->scale * dot(qi, K + j * J->d, J->d);
            if (s > M) M = s;
        }
    }
    /* pass 1b: row sum of shifted exponentials */
    double l = 0.0;
    for (int64_t j0 = 0; j0 < nvis; j0 += J->block) {
        int64_t j1 = j0 + J->block < nvis ? j0 + J->block : nvis;
        for (int64_t j = j0; j < j1; ++j)
            l += exp(J->scale * dot(qi, K + j * J->d, J->d) - M);
    }
    /* pass 2: normalised weights times values */
    for (int64_t j0 = 0; j0 < nvis; j0 += J->block) {
        int64_t j1 = j0 + J->block < nvis ? j0 + J->block : nvis;
        for (int64_t j = j0; j < j1; ++j) {
            double p = exp(J->scale * dot(qi, K + j * J->d, J->d) - M) / l;
            const double *vj = V + j * J->dv;
            for (int64_t c = 0; c < J->dv; ++c) oi[c] += p * vj[c];
        }
    }
    J->lse[bh * J->R + r] = M + log(l);
}

static void *worker(void *arg) {
    const job_t *J = (const job_t *)arg;
    for (int64_t r = J->row_begin; r < J->row_end; ++r) one_row(J, r / J->R, r % J->R);
    return NULL;
}

/* q, o, lse hold R rows per head: all Nq queries when rows == NULL (R = Nq),
 * else the queries rows[0..R-1] (each in [0, Nq)).  k, v hold Nk rows per head.
 * Returns 0 on success, -1 on bad arguments, -2 if memory for threads is missing. */
int oracle_twopass_fwd(const double *q, const double *k, const double *v, double *o, double *lse,
                       int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv, double scale,
                       int causal, const int64_t *rows, int64_t R, int64_t block, int nthreads) {
    if (!q || !k || !v || !o || !lse || BH < 0 || Nq < 0 || Nk < 0 || d < 1 || dv < 1 || block < 1)
        return -1;
    if (!rows) R = Nq;
    if (R < 0) return -1;
    if (rows)
        for (int64_t r = 0; r < R; ++r)
            if (rows[r] < 0 || rows[r] >= Nq) return -1;
    if (nthreads < 1) nthreads = 1;
    int64_t total = BH * R;
    if (total == 0) return 0;
    if (nthreads > total) nthreads = (int)total;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    char *live = (char *)calloc((size_t)nthreads, 1);
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)nthreads);
    if (!tid || !jobs || !live) {
        free(tid);
        free(live);
        free(jobs);
        return -2;
    }
    for (int t = 0; t < nthreads; ++t) {
        job_t J = {q, k, v, o, lse, BH, Nq, Nk, d, dv, scale, causal, block, rows, R,
                   total * t / nthreads, total * (t + 1) / nthreads};
        jobs[t] = J;
        if (pthread_create(&tid[t], NULL, worker, &jobs[t]) == 0)
            live[t] = 1;
        else
            worker(&jobs[t]); /* run inline if a thread cannot start */
    }
    for (int t = 0; t < nthreads; ++t)
        if (live[t]) pthread_join(tid[t], NULL);
    free(tid);
    free(live);
    free(jobs);
    return 0;
}
