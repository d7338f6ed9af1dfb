/*
 * ldn_oracle.c -- plain fp64 CPU oracle for the delta-rule linear-attention
 * family.  TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark call it; the product path never does.
 * It shares no code, header or constant with the CUDA library.
 *
 * What it computes: the token-by-token recurrence, exactly as the pages state
 * it, with nothing blocked, fused or reordered.
 *
 *   Notation (math orientation, column vectors): the fast-weight memory
 *   W ("S" on some pages) is d_v x d_k; kappa = k (the caller applies any
 *   feature map / normalisation), the output reads the UPDATED memory.
 *
 *   "Linear Attention Architectures: Mechanisms, Trade-offs, and Cross-Layer
 *    Routing" (reading notes):
 *     Sec. 2.1, Eq. 8          y_i = W_i q_i                   (read after write)
 *     Sec. 2.3, Eqs. 9-10, 14  DeltaNet:  vbar = W_{i-1} k,  r = v - vbar,
 *                              W_i = W_{i-1} + beta r k^T
 *     Sec. 2.4, Eqs. 15-17     Gated DeltaNet: decay first, then the error:
 *                              vbar = alpha W_{i-1} k,  r = v - vbar,
 *                              W_i = alpha W_{i-1} + beta r k^T
 *     Sec. 2.5, Eqs. 18-20     KDA: D = Diag(a) multiplies W on the RIGHT
 *                              (key-feature side): vbar = W_{i-1} D k,
 *                              W_i = W_{i-1} D + beta (v - vbar) k^T
 *     Sec. 2.6, Eqs. 21-24     Gated DeltaNet-2: the erase and the write get
 *                              their own gates: Wt = W_{i-1} D, e = b * k,
 *                              z = w * v (elementwise), r = z - Wt e,
 *                              W_i = Wt + r k^T (the outer product keeps k)
 *   "Reading notes: State reduction by key/query channel pruning",
 *     Sec. 2.1, Eqs. 1-2       the same DeltaNet update in S notation.
 *
 * Readings where the pages leave a step open:
 *   - gates arrive as natural-log decays g (alpha = exp(g), a_c = exp(g_c));
 *     the Mamba2-style parameterisation in the Residual Linear Attention notes
 *     (Sec. 2.2) produces exactly such a log value;
 *   - no query scale (the benchmark's method sources call the kernels with
 *     scale = 1);
 *   - the initial state is supplied and returned in memory orientation
 *     H = W^T, laid out [B][H][d_k][d_v] row-major ("K x V" state in the
 *     benchmark's method sources); a NULL initial state means zeros.
 *
 * Inputs are fp32 arrays (bf16 inputs are exactly representable in fp32);
 * every value is widened to double before use and all arithmetic is fp64.
 * Parallelism: independent (batch, head) pairs are spread over POSIX threads;
 * within a pair the recurrence runs strictly in token order.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define LDN_ORACLE_MODE_DELTANET 0
#define LDN_ORACLE_MODE_GDN 1
#define LDN_ORACLE_MODE_KDA 2
#define LDN_ORACLE_MODE_GDN2 3

typedef struct {
    const float *q, *k, *v, *beta, *gate, *S0;
    const float *erase, *write; /* Gated DeltaNet-2: b [B][T][H][dk], w [B][T][H][dv] */
    double *out, *S_final;
    int B, T, H, dk, dv, mode;
    int next_unit; /* shared work counter, protected by lock */
    pthread_mutex_t lock;
} job_t;

/* One (batch, head) pair: the recurrence over all T tokens. */
static void run_unit(const job_t *J, int unit, double *W, double *pred)
{
    const int b = unit / J->H, h = unit % J->H;
    const int dk = J->dk, dv = J->dv, H = J->H, T = J->T;

    /* W is d_v x d_k, row-major: W[i*dk + c]. */
    if (J->S0) {
        const float *s0 = J->S0 + ((size_t)b * H + h) * (size_t)dk * dv;
        for (int c = 0; c < dk; ++c)
            for (int i = 0; i < dv; ++i)
                W[(size_t)i * dk + c] = (double)s0[(size_t)c * dv + i];
    } else {
        memset(W, 0, sizeof(double) * (size_t)dk * dv);
    }

    for (int t = 0; t < T; ++t) {
        const size_t tok = ((size_t)b * T + t) * H + h; /* index of (b,t,h) */
        const float *q = J->q + tok * dk;
        const float *k = J->k + tok * dk;
        const float *v = J->v + tok * dv;
        const int gdn2 = J->mode == LDN_ORACLE_MODE_GDN2;
        const double beta = gdn2 ? 1.0 : (double)J->beta[tok];
        const float *eb = gdn2 ? J->erase + tok * dk : NULL;   /* e = b * k */
        const float *ww = gdn2 ? J->write + tok * dv : NULL;   /* z = w * v */

        /* Forget step: scalar alpha (Eqs. 15-17) or W <- W Diag(a) (Eqs. 18-20). */
        if (J->mode == LDN_ORACLE_MODE_GDN) {
            const double alpha = exp((double)J->gate[tok]);
            for (size_t e = 0; e < (size_t)dk * dv; ++e) W[e] *= alpha;
        } else if (J->mode == LDN_ORACLE_MODE_KDA || gdn2) {
            const float *g = J->gate + tok * dk;
            for (int c = 0; c < dk; ++c) {
                const double a = exp((double)g[c]);
                for (int i = 0; i < dv; ++i) W[(size_t)i * dk + c] *= a;
            }
        }

        /* Prediction of the (decayed) memory for the current key, Eq. 9
           (Gated DeltaNet-2: along the erase direction e = b * k, Eq. 23). */
        for (int i = 0; i < dv; ++i) {
            double s = 0.0;
            for (int c = 0; c < dk; ++c)
                s += W[(size_t)i * dk + c] * (gdn2 ? (double)eb[c] * (double)k[c] : (double)k[c]);
            pred[i] = s;
        }
        /* Write the error along the key, Eq. 10: W += beta (v - pred) k^T
           (Gated DeltaNet-2, Eq. 24: W += (w * v - pred) k^T). */
        for (int i = 0; i < dv; ++i) {
            const double target = gdn2 ? (double)ww[i] * (double)v[i] : (double)v[i];
            const double r = beta * (target - pred[i]);
            for (int c = 0; c < dk; ++c) W[(size_t)i * dk + c] += r * (double)k[c];
        }
        /* Read the updated memory with the query, Eq. 8. */
        double *o = J->out + tok * dv;
        for (int i = 0; i < dv; ++i) {
            double s = 0.0;
            for (int c = 0; c < dk; ++c) s += W[(size_t)i * dk + c] * (double)q[c];
            o[i] = s;
        }
    }

    if (J->S_final) {
        double *sf = J->S_final + ((size_t)b * H + h) * (size_t)dk * dv;
        for (int c = 0; c < dk; ++c)
            for (int i = 0; i < dv; ++i)
                sf[(size_t)c * dv + i] = W[(size_t)i * dk + c];
    }
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    double *W = (double *)malloc(sizeof(double) * (size_t)J->dk * J->dv);
    double *pred = (double *)malloc(sizeof(double) * (size_t)J->dv);
    if (!W || !pred) { free(W); free(pred); return (void *)1; }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int unit = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (unit >= J->B * J->H) break;
        run_unit(J, unit, W, pred);
    }
    free(W);
    free(pred);
    return NULL;
}

static int run_job(job_t *J, int nthreads, int *threads_used);

/* Number of host threads ldn_oracle_fwd uses for nthreads <= 0. */
int ldn_oracle_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * ldn_oracle_fwd: the whole recurrence for every (batch, head) pair.
 *   q, k   [B][T][H][dk]  fp32     v    [B][T][H][dv]  fp32
 *   beta   [B][T][H]      fp32     gate log-decay: mode 1 [B][T][H], mode 2
 *                                  [B][T][H][dk], mode 0 ignored (may be NULL)
 *   S0     [B][H][dk][dv] fp32 or NULL (zeros)
 *   out    [B][T][H][dv]  fp64     S_final [B][H][dk][dv] fp64 or NULL
 * Returns 0 on success, -1 on bad arguments, -2 on thread/alloc failure.
 * Returns the number of threads used through *threads_used when non-NULL.
 */
int ldn_oracle_fwd(const float *q, const float *k, const float *v,
                   const float *beta, const float *gate, const float *S0,
                   double *out, double *S_final,
                   int B, int T, int H, int dk, int dv, int mode,
                   int nthreads, int *threads_used)
{
    if (!q || !k || !v || !beta || !out) return -1;
    if (B < 0 || T < 0 || H < 0 || dk < 1 || dv < 1) return -1;
    if (mode < 0 || mode > 2) return -1;
    if (mode != LDN_ORACLE_MODE_DELTANET && !gate) return -1;

    job_t J;
    J.q = q; J.k = k; J.v = v; J.beta = beta; J.gate = gate; J.S0 = S0;
    J.erase = NULL; J.write = NULL;
    J.out = out; J.S_final = S_final;
    J.B = B; J.T = T; J.H = H; J.dk = dk; J.dv = dv; J.mode = mode;
    return run_job(&J, nthreads, threads_used);
}

/*
 * ldn_oracle_fwd_gdn2: the Gated DeltaNet-2 recurrence (Sec. 2.6, Eqs. 21-24)
 * for every (batch, head) pair.  As ldn_oracle_fwd, with the write strength
 * beta replaced by the erase gate b [B][T][H][dk] (e = b * k) and the write
 * gate w [B][T][H][dv] (z = w * v); gate is the per-key-channel log-decay
 * [B][T][H][dk].
 */
int ldn_oracle_fwd_gdn2(const float *q, const float *k, const float *v,
                        const float *erase, const float *write, const float *gate, const float *S0,
                        double *out, double *S_final, int B, int T, int H, int dk, int dv,
                        int nthreads, int *threads_used)
{
    if (!q || !k || !v || !erase || !write || !gate || !out) return -1;
    if (B < 0 || T < 0 || H < 0 || dk < 1 || dv < 1) return -1;
    job_t J;
    J.q = q; J.k = k; J.v = v; J.beta = NULL; J.gate = gate; J.S0 = S0;
    J.erase = erase; J.write = write;
    J.out = out; J.S_final = S_final;
    J.B = B; J.T = T; J.H = H; J.dk = dk; J.dv = dv; J.mode = LDN_ORACLE_MODE_GDN2;
    return run_job(&J, nthreads, threads_used);
}

static int run_job(job_t *J_, int nthreads, int *threads_used)
{
    job_t J = *J_;
    J.next_unit = 0;
    pthread_mutex_init(&J.lock, NULL);
    const int B = J.B, H = J.H;

    int units = B * H;
    if (nthreads <= 0) nthreads = ldn_oracle_default_threads();
    if (nthreads > units) nthreads = units > 0 ? units : 1;
    if (threads_used) *threads_used = nthreads;

    int rc = 0;
    if (units == 0) { pthread_mutex_destroy(&J.lock); return 0; }
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!tid) { pthread_mutex_destroy(&J.lock); return -2; }
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&tid[i], NULL, worker, &J) != 0) { rc = -2; break; }
        ++started;
    }
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(tid[i], &ret);
        if (ret) rc = -2;
    }
    free(tid);
    pthread_mutex_destroy(&J.lock);
    return rc;
}
