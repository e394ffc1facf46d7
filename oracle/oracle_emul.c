/*
 * Number-format emulation of attention — TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite loads this file's library (it is compiled into the
 * same liboracle.so as oracle_attn.c).  The product library never links,
 * includes or calls it, and this file includes nothing from the product.
 *
 * "Is Flash Attention Stable?" §III and §IV-A (Fig. 2, Fig. 3) describe a
 * numerical re-implementation of attention in which every step runs in a
 * chosen number format, from BF16 to FP64, so that FlashAttention and the
 * materialising baseline can be compared format by format; §IV-B (Fig. 6)
 * perturbs the algorithm's block sizes.  The pages give no code for it.
 * This file restates that instrument under one plain reading:
 *
 *   A format F has `mbits` fraction bits and `ebits` exponent bits (IEEE
 *   style: subnormals, round to nearest with ties to even, overflow to
 *   infinity).  fl(x) rounds an exact value to F.  Every tensor operation
 *   of the algorithm produces its result in F: elementwise operations are
 *   evaluated exactly (binary64) and rounded once; a reduction (row sum,
 *   row maximum) or a matrix product accumulates in binary64 and rounds
 *   its result once.  The inputs Q, K, V are first rounded to F.
 *
 *  oracle_round_fmt — fl(x), from the definition: the spacing of F near x
 *    is 2^(e - mbits), e being x's binary exponent clamped below at the
 *    smallest normal exponent; x is rounded to a multiple of that spacing,
 *    and a result above the largest finite value of F becomes infinite.
 *
 *  oracle_emul_rows — one output row per query row, with the steps of the
 *    chosen algorithm, each op rounded to F:
 *    scores   s_j = fl(scale * (q . k_j)), then fl(s_j + mask_j) when a key
 *             mask is given; -inf for a masked or (causal) future key.
 *    baseline the paper's "baseline attention" (§IV): P = fl(softmax(s))
 *             (one softmax op: maximum, exp, sum and division inside it),
 *             then O = fl(P V).
 *    tiled    FlashAttention's online merge (§II-B, Fig. 1; the running
 *             maximum m, denominator l and unnormalised output o of the
 *             yadro-code.ru tutorial), key blocks of width Bc in order:
 *               M  = max(m, max_j s_j), M' = (M == -inf ? 0 : M)
 *               a  = fl(exp(fl(m - M')))          (0 when m == -inf)
 *               p_j = fl(exp(fl(s_j - M')))
 *               l  = fl(fl(a * l) + fl(sum_j p_j))
 *               o  = fl(fl(a * o) + fl(sum_j p_j v_j))
 *             and at the end o = fl(o / l) (0 for a row with no allowed key).
 *    With F = binary64 both algorithms give softmax(QK^T*scale + mask)V up to
 *    binary64 rounding, which the tests check against oracle_attn_rows_f64.
 *
 *  oracle_emul_rows_planted — the same with one planted mistake, for the
 *    oracle's own tests only: `plant` names one rounding site above whose
 *    fl() is left out (or, for the last few, moved or duplicated).  The
 *    tests show that hand-worked rows in a coarse format tell every planted
 *    variant from the one above.  plant = 0 is oracle_emul_rows.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>

/* planted mistakes (test infrastructure): the rounding site that is changed */
enum {
    PLANT_NONE = 0,
    PLANT_Q_IN = 1,       /* Q used without rounding to F */
    PLANT_K_IN = 2,       /* K used without rounding to F */
    PLANT_V_IN = 3,       /* V used without rounding to F */
    PLANT_SCORE = 4,      /* scale * (q . k) not rounded */
    PLANT_MASK_ADD = 5,   /* s + mask not rounded */
    PLANT_M_DIFF = 6,     /* m - M' not rounded */
    PLANT_A_EXP = 7,      /* exp(m - M') not rounded */
    PLANT_S_DIFF = 8,     /* s_j - M' not rounded */
    PLANT_P_EXP = 9,      /* exp(s_j - M') not rounded */
    PLANT_AL = 10,        /* a * l not rounded */
    PLANT_ROWSUM = 11,    /* sum_j p_j of a block not rounded */
    PLANT_L_ADD = 12,     /* the sum a*l + rowsum not rounded */
    PLANT_AO = 13,        /* a * o not rounded */
    PLANT_PV = 14,        /* a block's P V not rounded */
    PLANT_O_ADD = 15,     /* the sum a*o + P V not rounded */
    PLANT_DIV = 16,       /* the final o / l not rounded */
    PLANT_L_LATE = 17,    /* l kept in binary64 and rounded once, at the end */
    PLANT_PV_PER_KEY = 18,/* P V rounded after every key instead of once per block */
    PLANT_DOT_PER_TERM = 19, /* q . k rounded after every term (a duplicated fl) */
    PLANT_SOFTMAX = 20,   /* baseline: P = softmax(s) not rounded */
    PLANT_BASE_PV = 21,   /* baseline: P V not rounded */
    PLANT_SOFTMAX_OPS = 22, /* baseline: exp, sum and division each rounded (three ops, not one) */
    PLANT_LAST = 22
};

double oracle_round_fmt(double x, int mbits, int ebits)
{
    if (x != x || isinf(x) || x == 0.0) return x;
    if (mbits >= 52 && ebits >= 11) return x; /* binary64 itself */
    const int emax = (1 << (ebits - 1)) - 1;  /* largest unbiased exponent */
    const int emin = 1 - emax;                /* smallest normal exponent */
    int e2;
    (void)frexp(fabs(x), &e2);                /* |x| = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                           /* exponent of x's leading bit */
    if (e < emin) e = emin;                   /* subnormals share one spacing */
    const double spacing = ldexp(1.0, e - mbits);
    double y = nearbyint(x / spacing) * spacing; /* ties to even */
    const double maxfinite = ldexp(2.0 - ldexp(1.0, -mbits), emax);
    if (fabs(y) > maxfinite) y = copysign(INFINITY, x);
    return y;
}

void oracle_round_array(const double *x, double *y, long long n, int mbits, int ebits)
{
    for (long long i = 0; i < n; ++i) y[i] = oracle_round_fmt(x[i], mbits, ebits);
}

typedef struct {
    const double *Q, *K, *V, *mask;
    int N, d, causal, algo, Bc, mbits, ebits, plant;
    double scale;
    const long long *rows;
    long long nrows;
    double *O;
    long long next;
    pthread_mutex_t lock;
    int fail;
} emul_job_t;

#define FL(v) oracle_round_fmt((v), job->mbits, job->ebits)
/* fl() at a named site: left out when that site is the planted one */
#define FLS(site, v) (job->plant == (site) ? (v) : FL(v))

/* scores of one query row, rounded as described above */
static void emul_scores(const emul_job_t *job, long long bh, int i, double *s)
{
    const int N = job->N, d = job->d;
    const double *q = job->Q + (bh * N + i) * (long long)d;
    for (int j = 0; j < N; ++j) {
        if (job->causal && j > i) {
            s[j] = -INFINITY;
            continue;
        }
        const double *k = job->K + (bh * N + j) * (long long)d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) {
            dot += FLS(PLANT_Q_IN, q[c]) * FLS(PLANT_K_IN, k[c]);
            if (job->plant == PLANT_DOT_PER_TERM) dot = FL(dot);
        }
        double x = FLS(PLANT_SCORE, job->scale * dot);
        if (job->mask) {
            const double mk = job->mask[bh * N + j];
            x = isinf(mk) && mk < 0 ? -INFINITY : FLS(PLANT_MASK_ADD, x + mk);
        }
        s[j] = x;
    }
}

static void emul_row(const emul_job_t *job, long long flat, double *s, double *p, double *o)
{
    const int N = job->N, d = job->d;
    const long long bh = flat / N;
    const int i = (int)(flat % N);
    const double *V = job->V + bh * N * (long long)d;
    emul_scores(job, bh, i, s);
    if (job->algo == 0) {
        /* baseline: one softmax op, then one matrix product */
        double mx = -INFINITY;
        for (int j = 0; j < N; ++j) mx = s[j] > mx ? s[j] : mx;
        if (mx == -INFINITY) {
            for (int c = 0; c < d; ++c) o[c] = 0.0;
            return;
        }
        const int ops = job->plant == PLANT_SOFTMAX_OPS;
        double sum = 0.0;
        for (int j = 0; j < N; ++j) {
            p[j] = ops ? FL(exp(FL(s[j] - mx))) : exp(s[j] - mx);
            sum += p[j];
        }
        if (ops) sum = FL(sum);
        for (int j = 0; j < N; ++j) p[j] = FLS(PLANT_SOFTMAX, p[j] / sum);
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int j = 0; j < N; ++j) acc += p[j] * FLS(PLANT_V_IN, V[(long long)j * d + c]);
            o[c] = FLS(PLANT_BASE_PV, acc);
        }
        return;
    }
    /* tiled: online merge over key blocks of width Bc */
    double m = -INFINITY, l = 0.0;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int j0 = 0; j0 < N; j0 += job->Bc) {
        const int j1 = j0 + job->Bc < N ? j0 + job->Bc : N;
        double mb = -INFINITY;
        for (int j = j0; j < j1; ++j) mb = s[j] > mb ? s[j] : mb;
        const double M = m > mb ? m : mb;
        const double Mu = (M == -INFINITY) ? 0.0 : M;
        const double a = (m == -INFINITY) ? 0.0 : FLS(PLANT_A_EXP, exp(FLS(PLANT_M_DIFF, m - Mu)));
        double rs = 0.0;
        for (int j = j0; j < j1; ++j) {
            p[j] = (s[j] == -INFINITY) ? 0.0 : FLS(PLANT_P_EXP, exp(FLS(PLANT_S_DIFF, s[j] - Mu)));
            rs += p[j];
        }
        if (job->plant == PLANT_L_LATE)
            l = a * l + rs;
        else
            l = FLS(PLANT_L_ADD, FLS(PLANT_AL, a * l) + FLS(PLANT_ROWSUM, rs));
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int j = j0; j < j1; ++j) {
                acc += p[j] * FLS(PLANT_V_IN, V[(long long)j * d + c]);
                if (job->plant == PLANT_PV_PER_KEY) acc = FL(acc);
            }
            o[c] = FLS(PLANT_O_ADD, FLS(PLANT_AO, a * o[c]) + FLS(PLANT_PV, acc));
        }
        m = M;
    }
    if (job->plant == PLANT_L_LATE) l = FL(l);
    for (int c = 0; c < d; ++c) o[c] = (l == 0.0) ? 0.0 : FLS(PLANT_DIV, o[c] / l);
}

static void *emul_worker(void *arg)
{
    emul_job_t *job = (emul_job_t *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)job->N);
    double *p = (double *)malloc(sizeof(double) * (size_t)job->N);
    if (!s || !p) {
        pthread_mutex_lock(&job->lock);
        job->fail = 1;
        pthread_mutex_unlock(&job->lock);
        free(s);
        free(p);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&job->lock);
        const long long r = job->next++;
        pthread_mutex_unlock(&job->lock);
        if (r >= job->nrows) break;
        const long long flat = job->rows ? job->rows[r] : r;
        emul_row(job, flat, s, p, job->O + r * job->d);
    }
    free(s);
    free(p);
    return NULL;
}

int oracle_emul_rows_planted(const double *Q, const double *K, const double *V, const double *mask, int BH,
                             int N, int d, int causal, double scale, int algo, int Bc, int mbits, int ebits,
                             const long long *rows, long long nrows, double *O, int nthreads, int plant)
{
    if (!Q || !K || !V || !O || BH <= 0 || N <= 0 || d <= 0 || Bc <= 0 || mbits < 1 || mbits > 52 ||
        ebits < 2 || ebits > 11 || (algo != 0 && algo != 1) || plant < 0 || plant > PLANT_LAST)
        return -1;
    if (rows)
        for (long long r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= (long long)BH * N) return -1;
    emul_job_t job;
    job.Q = Q;
    job.K = K;
    job.V = V;
    job.mask = mask;
    job.N = N;
    job.d = d;
    job.causal = causal;
    job.algo = algo;
    job.Bc = Bc;
    job.mbits = mbits;
    job.ebits = ebits;
    job.plant = plant;
    job.scale = scale;
    job.rows = rows;
    job.nrows = rows ? nrows : (long long)BH * N;
    job.O = O;
    job.next = 0;
    job.fail = 0;
    pthread_mutex_init(&job.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, emul_worker, &job) != 0) break;
        ++started;
    }
    if (started == 0) emul_worker(&job);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&job.lock);
    return job.fail ? -1 : 0;
}

int oracle_emul_rows(const double *Q, const double *K, const double *V, const double *mask, int BH, int N,
                     int d, int causal, double scale, int algo, int Bc, int mbits, int ebits,
                     const long long *rows, long long nrows, double *O, int nthreads)
{
    return oracle_emul_rows_planted(Q, K, V, mask, BH, N, d, causal, scale, algo, Bc, mbits, ebits, rows, nrows, O,
                                    nthreads, PLANT_NONE);
}
