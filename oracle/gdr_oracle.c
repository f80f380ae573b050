/*
 * gdr_oracle.c -- fp64 reference for the channelwise gated delta rule forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA library is
 * checked against.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load it.  It shares no code, header or constant
 * with the CUDA path under channelwise_gated_delta_gb300/csrc.
 *
 * What it computes (page "Reorder channelwise gated delta rule chunked hot
 * loops for autovectorization", pytorch/executorch PR #21021, first commit
 * summary): for every (batch b, value head hv) an fp64 state S[dk][dv]
 * (row i = key channel, column j = value channel) is carried over the tokens
 * in order, and each token does, as four separate sweeps over S:
 *
 *   1. decay      S[i][:]  *= exp(g_t[i])                 (per key channel)
 *   2. predict    vhat[j]   = sum_i S[i][j] * k_t[i]       (uses decayed S)
 *   3. update     S[i][j]  += beta_t * k_t[i] * (v_t[j] - vhat[j])
 *   4. output     o_t[j]    = sum_i S[i][j] * q_t[i]       (uses updated S)
 *
 * The PR reduces these four traversals to two for speed; the oracle keeps the
 * plain four-sweep form because it is the definition.  The chunked WY/UT form
 * of the second commit reaches the same result in exact arithmetic, so the
 * oracle is this definition and not that algorithm.
 *
 * Readings of points the page leaves open (each is a test-pinned choice):
 *   - g is a natural-log decay, one value per (token, value head, key channel);
 *   - beta is one scalar per (token, value head), used as given;
 *   - there is no 1/sqrt(dk) query scale;
 *   - grouped heads: value head hv reads key/query head hv / (HV / HK);
 *   - h0 == NULL means a zero initial state; ht == NULL means "not stored".
 *
 * Layouts (row-major, last index fastest):
 *   q, k   [B][T][HK][dk]      v, out [B][T][HV][dv]
 *   g      [B][T][HV][dk]      beta   [B][T][HV]
 *   h0, ht [B][HV][dk][dv]
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const double *q, *k, *v, *g, *beta, *h0;
    double *out, *ht;
    long B, T, HK, HV, dk, dv;
    long first_head, head_step; /* this worker takes heads first, first+step, ... */
    int status;
} oracle_job;

/* One (b, hv) pair over all its tokens. Returns 0, or 1 on allocation failure. */
static int run_head(const oracle_job *a, long b, long hv)
{
    const long dk = a->dk, dv = a->dv, T = a->T, HK = a->HK, HV = a->HV;
    const long group = HV / HK;
    const long hk = hv / group;
    double *S = (double *)calloc((size_t)(dk * dv), sizeof(double));
    double *vhat = (double *)calloc((size_t)dv, sizeof(double));
    if (!S || !vhat) {
        free(S);
        free(vhat);
        return 1;
    }
    if (a->h0) {
        memcpy(S, a->h0 + (b * HV + hv) * dk * dv, (size_t)(dk * dv) * sizeof(double));
    }
    for (long t = 0; t < T; ++t) {
        const double *qt = a->q + ((b * T + t) * HK + hk) * dk;
        const double *kt = a->k + ((b * T + t) * HK + hk) * dk;
        const double *vt = a->v + ((b * T + t) * HV + hv) * dv;
        const double *gt = a->g + ((b * T + t) * HV + hv) * dk;
        const double bt = a->beta[(b * T + t) * HV + hv];
        double *ot = a->out + ((b * T + t) * HV + hv) * dv;

        /* sweep 1: decay each key-channel row of the state */
        for (long i = 0; i < dk; ++i) {
            const double gamma = exp(gt[i]);
            for (long j = 0; j < dv; ++j) S[i * dv + j] *= gamma;
        }
        /* sweep 2: prediction from the decayed state, vhat = S^T k */
        for (long j = 0; j < dv; ++j) vhat[j] = 0.0;
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) vhat[j] += S[i * dv + j] * kt[i];
        /* sweep 3: rank-one delta update, S += beta k (v - vhat)^T */
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) S[i * dv + j] += bt * kt[i] * (vt[j] - vhat[j]);
        /* sweep 4: output from the updated state, o = S^T q */
        for (long j = 0; j < dv; ++j) ot[j] = 0.0;
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) ot[j] += S[i * dv + j] * qt[i];
    }
    if (a->ht) {
        memcpy(a->ht + (b * HV + hv) * dk * dv, S, (size_t)(dk * dv) * sizeof(double));
    }
    free(S);
    free(vhat);
    return 0;
}

static void *worker(void *p)
{
    oracle_job *a = (oracle_job *)p;
    const long heads = a->B * a->HV;
    for (long h = a->first_head; h < heads; h += a->head_step) {
        if (run_head(a, h / a->HV, h % a->HV)) {
            a->status = 1;
            return NULL;
        }
    }
    return NULL;
}

/* Number of online host cores (what "threads <= 0" resolves to). */
int gdr_oracle_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Runs the recurrence for every (b, hv), spread over `threads` POSIX threads
 * (<= 0: one per online core).  Returns 0 on success, 2 on a bad argument,
 * 1 on an allocation or thread failure.
 */
int gdr_oracle_f64(const double *q, const double *k, const double *v, const double *g,
                   const double *beta, const double *h0, double *out, double *ht,
                   long B, long T, long HK, long HV, long dk, long dv, int threads)
{
    if (B < 0 || T < 0 || HK <= 0 || HV <= 0 || dk <= 0 || dv <= 0 || HV % HK != 0) return 2;
    if ((B * T > 0) && (!q || !k || !v || !g || !beta || !out)) return 2;
    if (threads <= 0) threads = gdr_oracle_default_threads();
    const long heads = B * HV;
    if (heads == 0) return 0;
    if (threads > heads) threads = (int)heads;

    oracle_job *jobs = (oracle_job *)calloc((size_t)threads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return 1;
    }
    int status = 0;
    int started = 0;
    for (int w = 0; w < threads; ++w) {
        oracle_job j = {q, k, v, g, beta, h0, out, ht, B, T, HK, HV, dk, dv, w, threads, 0};
        jobs[w] = j;
        if (pthread_create(&tids[w], NULL, worker, &jobs[w]) != 0) {
            status = 1;
            break;
        }
        ++started;
    }
    for (int w = 0; w < started; ++w) {
        pthread_join(tids[w], NULL);
        if (jobs[w].status) status = 1;
    }
    free(jobs);
    free(tids);
    return status;
}
