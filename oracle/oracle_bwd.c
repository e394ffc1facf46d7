/*
 * FP64 CPU oracle for the gradients of exact attention — TEST
 * INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark load this file's library. The product library never links,
 * includes or calls it, and this file includes nothing from the product.
 *
 * What it computes (IEEE binary64, no blocking, no fusion): for
 *     O = softmax(Q K^T * scale + mask) V
 * ("Is Flash Attention Stable?" §II-A, the Attention(Q,K,V) equation) and an
 * upstream gradient dO = dL/dO, the gradients dL/dQ, dL/dK, dL/dV, by the
 * chain rule written out one query row at a time:
 *
 *   s_ij  = scale * <q_i, k_j> + mask_j   (-inf where causal j > i or masked)
 *   P_ij  = exp(s_ij - max_j s_ij) / sum_j exp(s_ij - max_j s_ij)
 *   G_ij  = dL/dP_ij = <dO_i, v_j>                 (O_i = sum_j P_ij v_j)
 *   dV_j += P_ij dO_i
 *   dS_ij = dL/ds_ij = P_ij (G_ij - sum_l P_il G_il)
 *                      (the Jacobian of the softmax: dP_ij/ds_il = P_ij (delta_jl - P_il))
 *   dQ_i  = scale * sum_j dS_ij k_j
 *   dK_j += scale * dS_ij q_i
 *
 * The yadro-code.ru FlashAttention tutorial notes that the backward pass of
 * the method recomputes intermediate values instead of storing them, and
 * that a check of an implementation compares gradients as well as outputs
 * within the tolerance of its number format; this file is that comparison's
 * reference.  It stores nothing it would not also recompute: each row's
 * scores are formed again from Q and K.  A fully masked row (O = 0, a
 * constant) contributes nothing.  The mask is a constant input: no gradient
 * is formed for it.
 *
 * `plant` is for the oracle's own tests: 1 drops the "- sum_l P_il G_il"
 * term of dS (the softmax Jacobian's rank-one part), 2 leaves out `scale`
 * in dQ and dK.  Both must fail the finite-difference pins.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>

typedef struct {
    const double *Q, *K, *V, *dO, *mask;
    int N, d, causal, plant;
    double scale;
    const long long *heads; /* NULL: heads 0 .. nheads-1 */
    long long nheads;
    double *dQ, *dK, *dV;   /* [nheads][N][d] */
    long long next;
    pthread_mutex_t lock;
    int fail;
} bwd_job_t;

static void bwd_head(const bwd_job_t *job, long long slot, double *s, double *P, double *G)
{
    const int N = job->N, d = job->d;
    const long long bh = job->heads ? job->heads[slot] : slot;
    const long long base = bh * (long long)N * d;
    const double *Qh = job->Q + base, *Kh = job->K + base, *Vh = job->V + base, *dOh = job->dO + base;
    const double *mk = job->mask ? job->mask + bh * (long long)N : NULL;
    double *dQ = job->dQ + slot * (long long)N * d;
    double *dK = job->dK + slot * (long long)N * d;
    double *dV = job->dV + slot * (long long)N * d;
    const double gscale = job->plant == 2 ? 1.0 : job->scale;

    for (long long e = 0; e < (long long)N * d; ++e) { dQ[e] = 0.0; dK[e] = 0.0; dV[e] = 0.0; }

    for (int i = 0; i < N; ++i) {
        const double *qi = Qh + (long long)i * d;
        const double *doi = dOh + (long long)i * d;
        /* scores and their maximum */
        double m = -INFINITY;
        for (int j = 0; j < N; ++j) {
            if (job->causal && j > i) { s[j] = -INFINITY; continue; }
            const double *kj = Kh + (long long)j * d;
            double dot = 0.0;
            for (int c = 0; c < d; ++c) dot += qi[c] * kj[c];
            double sj = job->scale * dot;
            if (mk) sj += mk[j];
            s[j] = sj;
            if (sj > m) m = sj;
        }
        if (m == -INFINITY) continue;          /* fully masked row: O_i = 0, constant */
        /* softmax row */
        double L = 0.0;
        for (int j = 0; j < N; ++j) {
            P[j] = s[j] == -INFINITY ? 0.0 : exp(s[j] - m);
            L += P[j];
        }
        for (int j = 0; j < N; ++j) P[j] /= L;
        /* G_ij = <dO_i, v_j> and its P-weighted mean */
        double c_i = 0.0;
        for (int j = 0; j < N; ++j) {
            if (P[j] == 0.0) { G[j] = 0.0; continue; }
            const double *vj = Vh + (long long)j * d;
            double dot = 0.0;
            for (int c = 0; c < d; ++c) dot += doi[c] * vj[c];
            G[j] = dot;
            c_i += P[j] * dot;
        }
        if (job->plant == 1) c_i = 0.0;
        /* accumulate the three gradients */
        double *dqi = dQ + (long long)i * d;
        for (int j = 0; j < N; ++j) {
            if (P[j] == 0.0) continue;
            const double dS = P[j] * (G[j] - c_i);
            const double *kj = Kh + (long long)j * d;
            double *dkj = dK + (long long)j * d;
            double *dvj = dV + (long long)j * d;
            for (int c = 0; c < d; ++c) {
                dvj[c] += P[j] * doi[c];
                dqi[c] += gscale * dS * kj[c];
                dkj[c] += gscale * dS * qi[c];
            }
        }
    }
}

static void *bwd_worker(void *arg)
{
    bwd_job_t *job = (bwd_job_t *)arg;
    const size_t n = (size_t)job->N;
    double *s = (double *)malloc(sizeof(double) * n);
    double *P = (double *)malloc(sizeof(double) * n);
    double *G = (double *)malloc(sizeof(double) * n);
    if (!s || !P || !G) {
        pthread_mutex_lock(&job->lock); job->fail = 1; pthread_mutex_unlock(&job->lock);
        free(s); free(P); free(G);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&job->lock);
        const long long h = job->next++;
        pthread_mutex_unlock(&job->lock);
        if (h >= job->nheads) break;
        bwd_head(job, h, s, P, G);
    }
    free(s); free(P); free(G);
    return NULL;
}

/*
 * Q, K, V, dO: [BH][N][d] row-major doubles.  key_mask: NULL or [BH][N]
 * additive (finite or -inf).  heads: NULL for every head (dQ, dK, dV are
 * then [BH][N][d]), else `nheads` head ids bh (outputs [nheads][N][d]).
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_attn_bwd_f64(const double *Q, const double *K, const double *V, const double *dO,
                        const double *key_mask, int BH, int N, int d, int causal, double scale,
                        const long long *heads, long long nheads, double *dQ, double *dK, double *dV,
                        int plant, int nthreads)
{
    if (!Q || !K || !V || !dO || !dQ || !dK || !dV || BH < 0 || N < 0 || d <= 0 || nheads < 0) return -1;
    if (!heads && nheads != BH) return -1;
    if (heads)
        for (long long h = 0; h < nheads; ++h)
            if (heads[h] < 0 || heads[h] >= BH) return -1;
    if (nheads == 0 || N == 0) return 0;
    bwd_job_t job;
    job.Q = Q; job.K = K; job.V = V; job.dO = dO; job.mask = key_mask;
    job.N = N; job.d = d; job.causal = causal; job.plant = plant; job.scale = scale;
    job.heads = heads; job.nheads = nheads;
    job.dQ = dQ; job.dK = dK; job.dV = dV;
    job.next = 0; job.fail = 0;
    pthread_mutex_init(&job.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nheads) nthreads = (int)nheads;
    if (nthreads > 256) nthreads = 256;
    pthread_t tid[256];
    int started = 0;
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&tid[started], NULL, bwd_worker, &job) == 0) ++started;
    bwd_worker(&job);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    pthread_mutex_destroy(&job.lock);
    return job.fail ? -1 : 0;
}
