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
 * Backward (ldn_oracle_bwd): the reverse-mode derivative of the same token
 * recurrence, step by step in reverse token order, from the full history of
 * decayed states Wt_t kept by a forward pass (the "first-order backward that
 * keeps the whole state history" the benchmark's method sources describe for
 * KDA).  For the loss L = sum_t <dO_t, o_t> + <dS_final, S_T> it returns the
 * gradient with respect to every input and the initial state.
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
    /* backward: upstream gradients (dS_final may be NULL) and the input gradients */
    const float *dout, *dS_final;
    double *dq, *dk_, *dv_, *dbeta, *dgate, *dS0;
    int bwd;
    int B, T, H, dk, dv, mode;
    int next_unit; /* shared work counter, protected by lock */
    pthread_mutex_t lock;
} job_t;

/* One (batch, head) pair: the recurrence over all T tokens.  Hist, when not
   NULL, receives the decayed state Wt of every token (T x dv x dk, for the
   backward); outputs are written only when J->out is set. */
static void run_unit(const job_t *J, int unit, double *W, double *pred, double *Hist)
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
        if (Hist) memcpy(Hist + (size_t)t * dk * dv, W, sizeof(double) * (size_t)dk * dv);

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
        if (!J->out) continue;
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

/*
 * One (batch, head) pair of the backward.  Forward, per token (as run_unit):
 *   Wt = W_{t-1} D_t          (D_t = alpha I, Diag(a), or I)
 *   p  = Wt k,  r = beta (v - p),  W_t = Wt + r k^T,  o = W_t q.
 * Reverse, with G = dL/dW_t (starting from dS_final^T):
 *   G += dO_t q^T                   dq_t  = W_t^T dO_t
 *   dr = G k                        dk_t  = G^T r + Wt^T dp,   dp = -beta dr
 *   dv_t = beta dr                  dbeta_t = dr . (v - p)
 *   Gt = G + dp k^T                 (gradient w.r.t. Wt)
 *   dg_t: KDA sum_i Gt[i][c] Wt[i][c] per channel c; GDN the sum over all
 *         entries (d alpha / d g = alpha, so these equal dL/dg)
 *   G <- Gt D_t                     (gradient w.r.t. W_{t-1})
 * and at the end dS0 = G^T.  Hist holds Wt for every token (T x dv x dk).
 */
static void run_unit_bwd(const job_t *J, int unit, double *Hist, double *W, double *G, double *r, double *e,
                         double *dp)
{
    const int b = unit / J->H, h = unit % J->H;
    const int dk = J->dk, dv = J->dv, H = J->H, T = J->T;
    const size_t D2 = (size_t)dk * dv;

    /* forward, keeping Wt of every token (outputs not written: J->out is NULL) */
    run_unit(J, unit, W, r, Hist);
    /* reverse */
    if (J->dS_final) {
        const float *sf = J->dS_final + ((size_t)b * H + h) * D2;
        for (int c = 0; c < dk; ++c)
            for (int i = 0; i < dv; ++i) G[(size_t)i * dk + c] = (double)sf[(size_t)c * dv + i];
    } else {
        memset(G, 0, sizeof(double) * D2);
    }
    for (int t = T - 1; t >= 0; --t) {
        const size_t tok = ((size_t)b * T + t) * H + h;
        const float *q = J->q + tok * dk, *k = J->k + tok * dk, *v = J->v + tok * dv;
        const float *dO = J->dout + tok * dv;
        const double beta = (double)J->beta[tok];
        const double *Wt = Hist + (size_t)t * D2;
        /* r and v - p of this token, and W_t = Wt + r k^T */
        for (int i = 0; i < dv; ++i) {
            double p = 0.0;
            for (int c = 0; c < dk; ++c) p += Wt[(size_t)i * dk + c] * (double)k[c];
            e[i] = (double)v[i] - p;
            r[i] = beta * e[i];
        }
        for (int i = 0; i < dv; ++i)
            for (int c = 0; c < dk; ++c) W[(size_t)i * dk + c] = Wt[(size_t)i * dk + c] + r[i] * (double)k[c];
        /* output read: G += dO q^T, dq = W_t^T dO */
        double *dq = J->dq + tok * dk;
        for (int c = 0; c < dk; ++c) {
            double s = 0.0;
            for (int i = 0; i < dv; ++i) s += W[(size_t)i * dk + c] * (double)dO[i];
            dq[c] = s;
        }
        for (int i = 0; i < dv; ++i)
            for (int c = 0; c < dk; ++c) G[(size_t)i * dk + c] += (double)dO[i] * (double)q[c];
        /* write W_t = Wt + r k^T */
        double *dkk = J->dk_ + tok * dk, *dvv = J->dv_ + tok * dv;
        double db = 0.0;
        for (int i = 0; i < dv; ++i) {
            double dr = 0.0;
            for (int c = 0; c < dk; ++c) dr += G[(size_t)i * dk + c] * (double)k[c];
            dvv[i] = beta * dr;
            db += dr * e[i];
            dp[i] = -beta * dr;
        }
        J->dbeta[tok] = db;
        for (int c = 0; c < dk; ++c) {
            double s = 0.0;
            for (int i = 0; i < dv; ++i) s += G[(size_t)i * dk + c] * r[i] + Wt[(size_t)i * dk + c] * dp[i];
            dkk[c] = s;
        }
        /* prediction p = Wt k: G <- G + dp k^T is the gradient w.r.t. Wt */
        for (int i = 0; i < dv; ++i)
            for (int c = 0; c < dk; ++c) G[(size_t)i * dk + c] += dp[i] * (double)k[c];
        /* decay Wt = W_{t-1} D_t */
        if (J->mode == LDN_ORACLE_MODE_GDN) {
            double s = 0.0;
            for (size_t x = 0; x < D2; ++x) s += G[x] * Wt[x];
            J->dgate[tok] = s;
            const double a_t = exp((double)J->gate[tok]);   /* alpha of this token */
            for (size_t x = 0; x < D2; ++x) G[x] *= a_t;
        } else if (J->mode == LDN_ORACLE_MODE_KDA) {
            const float *g = J->gate + tok * dk;
            double *dg = J->dgate + tok * dk;
            for (int c = 0; c < dk; ++c) {
                double s = 0.0;
                for (int i = 0; i < dv; ++i) s += G[(size_t)i * dk + c] * Wt[(size_t)i * dk + c];
                dg[c] = s;
                const double a = exp((double)g[c]);
                for (int i = 0; i < dv; ++i) G[(size_t)i * dk + c] *= a;
            }
        }
    }
    double *ds0 = J->dS0 + ((size_t)b * H + h) * D2;
    for (int c = 0; c < dk; ++c)
        for (int i = 0; i < dv; ++i) ds0[(size_t)c * dv + i] = G[(size_t)i * dk + c];
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    const size_t D2 = (size_t)J->dk * J->dv;
    double *W = (double *)malloc(sizeof(double) * D2);
    double *pred = (double *)malloc(sizeof(double) * (size_t)J->dv);
    double *G = J->bwd ? (double *)malloc(sizeof(double) * D2) : NULL;
    double *e = J->bwd ? (double *)malloc(sizeof(double) * (size_t)J->dv) : NULL;
    double *dp = J->bwd ? (double *)malloc(sizeof(double) * (size_t)J->dv) : NULL;
    double *Hist = J->bwd ? (double *)malloc(sizeof(double) * D2 * (size_t)(J->T > 0 ? J->T : 1)) : NULL;
    if (!W || !pred || (J->bwd && (!G || !e || !dp || !Hist))) {
        free(W); free(pred); free(G); free(e); free(dp); free(Hist);
        return (void *)1;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int unit = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (unit >= J->B * J->H) break;
        if (J->bwd)
            run_unit_bwd(J, unit, Hist, W, G, pred, e, dp);
        else
            run_unit(J, unit, W, pred, NULL);
    }
    free(W); free(pred); free(G); free(e); free(dp); free(Hist);
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
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.beta = beta; J.gate = gate; J.S0 = S0;
    J.out = out; J.S_final = S_final;
    J.B = B; J.T = T; J.H = H; J.dk = dk; J.dv = dv; J.mode = mode;
    return run_job(&J, nthreads, threads_used);
}

/*
 * ldn_oracle_bwd: gradients of L = sum <dout, o> + <dS_final, S_T> for modes
 * 0-2 (DeltaNet, Gated DeltaNet, KDA).  Inputs as ldn_oracle_fwd, plus
 *   dout    [B][T][H][dv] fp32     dS_final [B][H][dk][dv] fp32 or NULL (zero)
 * Outputs (fp64): dq, dk [B][T][H][dk], dv [B][T][H][dv], dbeta [B][T][H],
 *   dgate: mode 1 [B][T][H], mode 2 [B][T][H][dk], mode 0 not written (may be
 *   NULL); dS0 [B][H][dk][dv] (also when S0 is NULL: the gradient at zero).
 * Memory: T x dk x dv doubles per thread for the state history.
 */
int ldn_oracle_bwd(const float *q, const float *k, const float *v, const float *beta, const float *gate,
                   const float *S0, const float *dout, const float *dS_final, double *dq, double *dk_,
                   double *dv_, double *dbeta, double *dgate, double *dS0, int B, int T, int H, int dk, int dv,
                   int mode, int nthreads, int *threads_used)
{
    if (!q || !k || !v || !beta || !dout || !dq || !dk_ || !dv_ || !dbeta || !dS0) return -1;
    if (B < 0 || T < 0 || H < 0 || dk < 1 || dv < 1) return -1;
    if (mode < 0 || mode > 2) return -1;
    if (mode != LDN_ORACLE_MODE_DELTANET && (!gate || !dgate)) return -1;
    job_t J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.beta = beta; J.gate = gate; J.S0 = S0;
    J.dout = dout; J.dS_final = dS_final;
    J.dq = dq; J.dk_ = dk_; J.dv_ = dv_; J.dbeta = dbeta; J.dgate = dgate; J.dS0 = dS0;
    J.bwd = 1;
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
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.beta = NULL; J.gate = gate; J.S0 = S0;
    J.erase = erase; J.write = write;
    J.out = out; J.S_final = S_final;
    J.B = B; J.T = T; J.H = H; J.dk = dk; J.dv = dv; J.mode = LDN_ORACLE_MODE_GDN2;
    return run_job(&J, nthreads, threads_used);
}

/*
 * Residual Linear Attention (RLA) and Residual DeltaNet (RDN), "Residual Linear
 * Attention" reading notes, Sec. 2.2 (the boxed final form) and Sec. 2.4.  Per
 * token, with alpha = exp(gate) and the base state W and residual state R both
 * d_v x d_k:
 *   r  = Clip_[-c, c](v - W_{t-1} k)        (the OLD base state, neither decayed
 *                                            nor written yet; c = INFINITY: no clip)
 *   o  = alpha W_{t-1} q + gamma R_t q      (the UPDATED residual state)
 *   RLA: R_t = alpha R_{t-1} + gamma r k^T,  W_t = alpha W_{t-1} + beta v k^T
 *   RDN: R_t = alpha R_{t-1} (I - gamma k k^T) + gamma r k^T,
 *        W_t = alpha W_{t-1} (I - beta k k^T) + beta v k^T
 * The order follows the notes' pseudo-code: residual from the old base state,
 * update R, output, update W.
 */
typedef struct {
    const float *q, *k, *v, *beta, *gamma, *gate, *S0, *R0;
    float clip;
    int delta;   /* 0: RLA (additive updates), 1: RDN (delta updates) */
    double *out, *S_final, *R_final;
    int B, T, H, dk, dv;
    int next_unit;
    pthread_mutex_t lock;
} rla_job_t;

static void rla_unit(const rla_job_t *J, int unit, double *W, double *R, double *tmp)
{
    const int b = unit / J->H, h = unit % J->H;
    const int dk = J->dk, dv = J->dv, H = J->H, T = J->T;
    const size_t D2 = (size_t)dk * dv;
    const float *init[2] = {J->S0, J->R0};
    double *st[2] = {W, R};
    for (int m = 0; m < 2; ++m) {
        if (init[m]) {
            const float *s0 = init[m] + ((size_t)b * H + h) * D2;
            for (int c = 0; c < dk; ++c)
                for (int i = 0; i < dv; ++i) st[m][(size_t)i * dk + c] = (double)s0[(size_t)c * dv + i];
        } else {
            memset(st[m], 0, sizeof(double) * D2);
        }
    }
    const double clip = (double)J->clip;
    for (int t = 0; t < T; ++t) {
        const size_t tok = ((size_t)b * T + t) * H + h;
        const float *q = J->q + tok * dk, *k = J->k + tok * dk, *v = J->v + tok * dv;
        const double alpha = exp((double)J->gate[tok]), beta = (double)J->beta[tok], gamma = (double)J->gamma[tok];
        double *o = J->out + tok * dv;
        /* residual against the old base state; base read alpha W_{t-1} q into o */
        for (int i = 0; i < dv; ++i) {
            double pk = 0.0, sq = 0.0;
            for (int c = 0; c < dk; ++c) {
                pk += W[(size_t)i * dk + c] * (double)k[c];
                sq += W[(size_t)i * dk + c] * (double)q[c];
            }
            double r = (double)v[i] - pk;
            if (r > clip) r = clip;
            if (r < -clip) r = -clip;
            tmp[i] = r;
            o[i] = alpha * sq;
        }
        /* residual state */
        for (int i = 0; i < dv; ++i) {
            double rk = 0.0;
            for (int c = 0; c < dk; ++c) rk += R[(size_t)i * dk + c] * (double)k[c];
            const double w = gamma * (tmp[i] - (J->delta ? alpha * rk : 0.0));
            for (int c = 0; c < dk; ++c) R[(size_t)i * dk + c] = alpha * R[(size_t)i * dk + c] + w * (double)k[c];
        }
        /* output: alpha W_{t-1} q + gamma R_t q */
        for (int i = 0; i < dv; ++i) {
            double rq = 0.0;
            for (int c = 0; c < dk; ++c) rq += R[(size_t)i * dk + c] * (double)q[c];
            o[i] += gamma * rq;
        }
        /* base state */
        for (int i = 0; i < dv; ++i) {
            double wk = 0.0;
            for (int c = 0; c < dk; ++c) wk += W[(size_t)i * dk + c] * (double)k[c];
            const double w = beta * ((double)v[i] - (J->delta ? alpha * wk : 0.0));
            for (int c = 0; c < dk; ++c) W[(size_t)i * dk + c] = alpha * W[(size_t)i * dk + c] + w * (double)k[c];
        }
    }
    double *fin[2] = {J->S_final, J->R_final};
    for (int m = 0; m < 2; ++m) {
        if (!fin[m]) continue;
        double *sf = fin[m] + ((size_t)b * H + h) * D2;
        for (int c = 0; c < dk; ++c)
            for (int i = 0; i < dv; ++i) sf[(size_t)c * dv + i] = st[m][(size_t)i * dk + c];
    }
}

static void *rla_worker(void *arg)
{
    rla_job_t *J = (rla_job_t *)arg;
    const size_t D2 = (size_t)J->dk * J->dv;
    double *W = (double *)malloc(sizeof(double) * D2), *R = (double *)malloc(sizeof(double) * D2);
    double *tmp = (double *)malloc(sizeof(double) * (size_t)J->dv);
    if (!W || !R || !tmp) { free(W); free(R); free(tmp); return (void *)1; }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int unit = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (unit >= J->B * J->H) break;
        rla_unit(J, unit, W, R, tmp);
    }
    free(W); free(R); free(tmp);
    return NULL;
}

/*
 * ldn_oracle_rla: RLA (delta = 0) or RDN (delta = 1) for every (batch, head).
 *   q, k [B][T][H][dk]; v [B][T][H][dv]; beta, gamma, gate (log alpha) [B][T][H];
 *   clip c > 0 (INFINITY: none); S0, R0 [B][H][dk][dv] or NULL (zeros).
 *   out [B][T][H][dv] fp64; S_final, R_final [B][H][dk][dv] fp64 or NULL.
 */
int ldn_oracle_rla(const float *q, const float *k, const float *v, const float *beta, const float *gamma,
                   const float *gate, float clip, const float *S0, const float *R0, double *out, double *S_final,
                   double *R_final, int B, int T, int H, int dk, int dv, int delta, int nthreads)
{
    if (!q || !k || !v || !beta || !gamma || !gate || !out) return -1;
    if (B < 0 || T < 0 || H < 0 || dk < 1 || dv < 1 || !(clip > 0.0f)) return -1;
    rla_job_t J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.beta = beta; J.gamma = gamma; J.gate = gate; J.S0 = S0; J.R0 = R0;
    J.clip = clip; J.delta = delta ? 1 : 0;
    J.out = out; J.S_final = S_final; J.R_final = R_final;
    J.B = B; J.T = T; J.H = H; J.dk = dk; J.dv = dv;
    pthread_mutex_init(&J.lock, NULL);
    const int units = B * H;
    if (nthreads <= 0) nthreads = ldn_oracle_default_threads();
    if (nthreads > units) nthreads = units > 0 ? units : 1;
    int rc = 0;
    if (units > 0) {
        pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        if (!tid) { pthread_mutex_destroy(&J.lock); return -2; }
        int started = 0;
        for (int i = 0; i < nthreads; ++i) {
            if (pthread_create(&tid[i], NULL, rla_worker, &J) != 0) { rc = -2; break; }
            ++started;
        }
        for (int i = 0; i < started; ++i) {
            void *ret = NULL;
            pthread_join(tid[i], &ret);
            if (ret) rc = -2;
        }
        free(tid);
    }
    pthread_mutex_destroy(&J.lock);
    return rc;
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
