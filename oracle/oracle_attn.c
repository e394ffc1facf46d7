/*
 * FP64 CPU oracle for exact attention — TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark load this file's library. The product library never links,
 * includes or calls it, and this file includes nothing from the product.
 *
 * What it computes (all in IEEE binary64, no blocking, no fusion):
 *
 *  oracle_attn_rows_f64  — the definition of attention,
 *      O = softmax(Q K^T * scale + mask) V,
 *    from "Is Flash Attention Stable?" §II-A (the Attention(Q,K,V) equation
 *    with the 1/sqrt(d_k) factor passed in as `scale`), written out one query
 *    row at a time: scores, then the row maximum, then exp(s - max), the sum,
 *    and the weighted sum of V rows divided by that sum.  The maximum is
 *    subtracted before exponentiating because, as the yadro-code.ru tutorial
 *    on FlashAttention ("exact attention memory IO", the paragraph on the
 *    direct stable form) explains, that keeps every exponent <= 1 without
 *    changing the ratio.  Causal masking is top-left aligned: query i sees
 *    keys j <= i (the same tutorial's worked example, where each causal
 *    prefix is the set of allowed positions of a row).  A row with no
 *    allowed key (every score -inf) is left undefined by the tutorial; here
 *    it is defined as O = 0, LSE = -inf.  LSE is the natural-log
 *    log-sum-exp of the row's scaled, masked scores.
 *
 *  oracle_attn_rows_bs_f64 — the same definition with a block mask: the
 *    yadro-code.ru tutorial mentions that the method's paper also treats a
 *    block-sparse extension; read plainly, a block mask marks which
 *    (query block, key block) pairs of the score matrix take part, and every
 *    score outside the marked blocks is -inf before the softmax (a block row
 *    with no marked block is a fully masked row).  Blocks are `bq` query rows
 *    by `bk` keys; the mask is [BH][ceil(N/bq)][ceil(N/bk)] bytes, non-zero =
 *    take part.
 *
 *  oracle_blocked_row_f64 — the online merge for one row of scores,
 *    following the same tutorial's description of the running state
 *    (maximum m, denominator l, unnormalised vector a): when a block with a
 *    larger maximum M arrives, l and a are multiplied by exp(m - M) before
 *    the block's terms, taken relative to M, are added; the result is a / l
 *    at the end.  The initial maximum is -inf, which zeroes the not yet
 *    existing old sum.  Used only by the oracle's own self-tests (the blocked
 *    result must equal the direct one).  ORACLE_NO_RESCALE drops the
 *    exp(m - M) factor: the planted mistake of the tutorial's exercise,
 *    which the tests require to fail.
 *
 *  oracle_deviation_f64 — the deviation measures of the paper's §IV-A and
 *    §V: element-wise maximum absolute difference, and the 1-D
 *    Wasserstein-1 distance between the empirical value distributions of
 *    two equal-length tensors, (1/n) * sum_i |sort(a)_i - sort(b)_i|
 *    (the pages name the measure but their formula did not survive
 *    extraction; this is its standard definition for equal-weight samples).
 *    Also the mean and population standard deviation of |a - b| and the
 *    signed mean of a - b.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_NO_RESCALE 1

/* ------------------------------------------------------------------ */
/* Direct attention, one query row                                     */
/* ------------------------------------------------------------------ */

typedef struct {
    const double *Q, *K, *V, *mask;
    const unsigned char *bmask; /* NULL, or [BH][ceil(N/bq)][ceil(N/bk)] */
    int bq, bk;
    int N, d, causal;
    double scale;
    const long long *rows; /* NULL: rows 0 .. nrows-1 */
    long long nrows;
    double *O, *LSE;
    long long next;        /* shared work counter */
    pthread_mutex_t lock;
    int fail;
} rows_job_t;

static void direct_row(const rows_job_t *job, long long flat, double *s, double *o_out, double *lse_out)
{
    const int N = job->N, d = job->d;
    const long long bh = flat / N;
    const int i = (int)(flat % N);
    const double *q = job->Q + flat * d;
    const double *Kh = job->K + bh * (long long)N * d;
    const double *Vh = job->V + bh * (long long)N * d;
    const double *mk = job->mask ? job->mask + bh * (long long)N : NULL;
    const int nqb = job->bmask ? (N + job->bq - 1) / job->bq : 0;
    const int nkb = job->bmask ? (N + job->bk - 1) / job->bk : 0;
    const unsigned char *brow = job->bmask ? job->bmask + ((long long)bh * nqb + i / job->bq) * nkb : NULL;

    /* scores s_j = scale * <q_i, k_j> + mask_j, -inf where not allowed */
    double m = -INFINITY;
    for (int j = 0; j < N; ++j) {
        if (job->causal && j > i) { s[j] = -INFINITY; continue; }
        if (brow && !brow[j / job->bk]) { s[j] = -INFINITY; continue; }
        double dot = 0.0;
        const double *kj = Kh + (long long)j * d;
        for (int c = 0; c < d; ++c) dot += q[c] * kj[c];
        double sj = job->scale * dot;
        if (mk) sj += mk[j];
        s[j] = sj;
        if (sj > m) m = sj;
    }
    if (m == -INFINITY) {            /* fully masked row: defined as 0 */
        for (int c = 0; c < d; ++c) o_out[c] = 0.0;
        *lse_out = -INFINITY;
        return;
    }
    double L = 0.0;
    for (int c = 0; c < d; ++c) o_out[c] = 0.0;
    for (int j = 0; j < N; ++j) {
        if (s[j] == -INFINITY) continue;
        const double w = exp(s[j] - m);
        L += w;
        const double *vj = Vh + (long long)j * d;
        for (int c = 0; c < d; ++c) o_out[c] += w * vj[c];
    }
    for (int c = 0; c < d; ++c) o_out[c] /= L;
    *lse_out = m + log(L);
}

static void *rows_worker(void *arg)
{
    rows_job_t *job = (rows_job_t *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)job->N);
    if (!s) { pthread_mutex_lock(&job->lock); job->fail = 1; pthread_mutex_unlock(&job->lock); return NULL; }
    const long long chunk = 16;
    for (;;) {
        pthread_mutex_lock(&job->lock);
        long long r0 = job->next;
        job->next += chunk;
        pthread_mutex_unlock(&job->lock);
        if (r0 >= job->nrows) break;
        long long r1 = r0 + chunk < job->nrows ? r0 + chunk : job->nrows;
        for (long long r = r0; r < r1; ++r) {
            long long flat = job->rows ? job->rows[r] : r;
            direct_row(job, flat, s, job->O + r * job->d, job->LSE + r);
        }
    }
    free(s);
    return NULL;
}

/*
 * Q, K, V: [BH][N][d] row-major doubles.  key_mask: NULL or [BH][N] additive
 * (finite or -inf).  rows: NULL to compute every row (O is then [BH*N][d],
 * LSE [BH*N]), else `nrows` flat row ids bh*N + i (O is [nrows][d]).
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_attn_rows_bs_f64(const double *Q, const double *K, const double *V,
                            const double *key_mask, const unsigned char *block_mask, int bq, int bk,
                            int BH, int N, int d, int causal, double scale,
                            const long long *rows, long long nrows, double *O, double *LSE, int nthreads);

int oracle_attn_rows_f64(const double *Q, const double *K, const double *V,
                         const double *key_mask, int BH, int N, int d, int causal,
                         double scale, const long long *rows, long long nrows,
                         double *O, double *LSE, int nthreads)
{
    return oracle_attn_rows_bs_f64(Q, K, V, key_mask, NULL, 1, 1, BH, N, d, causal, scale, rows, nrows,
                                   O, LSE, nthreads);
}

/* As oracle_attn_rows_f64, with an optional block mask (NULL: none) of
 * bq x bk blocks. */
int oracle_attn_rows_bs_f64(const double *Q, const double *K, const double *V,
                            const double *key_mask, const unsigned char *block_mask, int bq, int bk,
                            int BH, int N, int d, int causal, double scale,
                            const long long *rows, long long nrows, double *O, double *LSE, int nthreads)
{
    if (block_mask && (bq <= 0 || bk <= 0)) return -1;
    if (!Q || !K || !V || !O || !LSE || BH <= 0 || N <= 0 || d <= 0) return -1;
    if (!rows) nrows = (long long)BH * N;
    for (long long r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= (long long)BH * N) return -1;
    rows_job_t job;
    memset(&job, 0, sizeof(job));
    job.Q = Q; job.K = K; job.V = V; job.mask = key_mask;
    job.bmask = block_mask; job.bq = bq; job.bk = bk;
    job.N = N; job.d = d; job.causal = causal; job.scale = scale;
    job.rows = rows; job.nrows = nrows; job.O = O; job.LSE = LSE;
    pthread_mutex_init(&job.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    int started = 0;
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&th[started], NULL, rows_worker, &job) == 0) ++started;
    rows_worker(&job);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&job.lock);
    return job.fail ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* Online (blocked) merge for one row of precomputed scores            */
/* ------------------------------------------------------------------ */

/*
 * scores: n values; values: [n][dv].  Blocks are [b*width, (b+1)*width).
 * block_order: NULL for natural order, else a permutation of the block
 * indices 0 .. ceil(n/width)-1 giving the order in which blocks are merged.
 * out: dv values a/l; lse_out (nullable): m + log(l).
 */
int oracle_blocked_row_f64(const double *scores, const double *values, int n, int dv,
                           int width, const int *block_order, int flags,
                           double *out, double *lse_out)
{
    if (!scores || !values || !out || n <= 0 || dv <= 0 || width <= 0) return -1;
    const int nblocks = (n + width - 1) / width;
    double m = -INFINITY, l = 0.0;
    double *a = (double *)calloc((size_t)dv, sizeof(double));
    if (!a) return -1;
    for (int bi = 0; bi < nblocks; ++bi) {
        const int b = block_order ? block_order[bi] : bi;
        if (b < 0 || b >= nblocks) { free(a); return -1; }
        const int j0 = b * width, j1 = (j0 + width < n) ? j0 + width : n;
        double M = m;
        for (int j = j0; j < j1; ++j) if (scores[j] > M) M = scores[j];
        /* bring the old sums to the new reference maximum M */
        if (!(flags & ORACLE_NO_RESCALE)) {
            const double r = (M == -INFINITY) ? 1.0 : exp(m - M);
            l *= r;
            for (int c = 0; c < dv; ++c) a[c] *= r;
        }
        for (int j = j0; j < j1; ++j) {
            if (scores[j] == -INFINITY) continue;
            const double w = exp(scores[j] - M);
            l += w;
            for (int c = 0; c < dv; ++c) a[c] += w * values[(long long)j * dv + c];
        }
        m = M;
    }
    if (l == 0.0) {
        for (int c = 0; c < dv; ++c) out[c] = 0.0;
        if (lse_out) *lse_out = -INFINITY;
    } else {
        for (int c = 0; c < dv; ++c) out[c] = a[c] / l;
        if (lse_out) *lse_out = m + log(l);
    }
    free(a);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Deviation measures                                                  */
/* ------------------------------------------------------------------ */

static int cmp_double(const void *x, const void *y)
{
    const double a = *(const double *)x, b = *(const double *)y;
    return (a > b) - (a < b);
}

/*
 * out[0] = max_i |a_i - b_i|
 * out[1] = W1 = (1/n) sum_i |sort(a)_i - sort(b)_i|
 * out[2] = mean |a_i - b_i|
 * out[3] = population std of |a_i - b_i|
 * out[4] = mean (a_i - b_i)
 * Pairs where both sides are the same infinity count as difference 0.
 */
int oracle_deviation_f64(const double *a, const double *b, long long n, double *out)
{
    if (!a || !b || !out || n <= 0) return -1;
    double mx = 0.0, s = 0.0, sd = 0.0;
    for (long long i = 0; i < n; ++i) {
        const double diff = (a[i] == b[i]) ? 0.0 : a[i] - b[i];
        const double ad = fabs(diff);
        if (ad > mx || isnan(ad)) mx = ad;
        s += ad;
        sd += diff;
    }
    const double mean = s / (double)n;
    double var = 0.0;                 /* second pass: sum of squared deviations */
    for (long long i = 0; i < n; ++i) {
        const double ad = (a[i] == b[i]) ? 0.0 : fabs(a[i] - b[i]);
        var += (ad - mean) * (ad - mean);
    }
    var /= (double)n;
    double *sa = (double *)malloc(sizeof(double) * (size_t)n);
    double *sb = (double *)malloc(sizeof(double) * (size_t)n);
    if (!sa || !sb) { free(sa); free(sb); return -1; }
    memcpy(sa, a, sizeof(double) * (size_t)n);
    memcpy(sb, b, sizeof(double) * (size_t)n);
    qsort(sa, (size_t)n, sizeof(double), cmp_double);
    qsort(sb, (size_t)n, sizeof(double), cmp_double);
    double w = 0.0;
    for (long long i = 0; i < n; ++i) w += (sa[i] == sb[i]) ? 0.0 : fabs(sa[i] - sb[i]);
    free(sa);
    free(sb);
    out[0] = mx;
    out[1] = w / (double)n;
    out[2] = mean;
    out[3] = sqrt(var);
    out[4] = sd / (double)n;
    return 0;
}
