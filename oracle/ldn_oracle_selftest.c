/*
 * ldn_oracle_selftest.c -- native self-test of the fp64 oracle (ldn_oracle.c).
 * TEST INFRASTRUCTURE ONLY, like the oracle itself: built beside it with gcc
 * and run by the CPU test suite, so that the oracle is checked without numpy
 * on whichever host compiled it.
 *
 * Each check compares the oracle with something other than its own loop:
 *   1. the worked example of the linear-attention notes (Sec. 2.3, DeltaNet):
 *      a unit key whose prediction is 2, target 5, beta 0.5 -> prediction 3.5,
 *      the orthogonal direction keeps its prediction;
 *   2. the exact write: beta = 1 with exactly unit (axis) keys stores v_t under
 *      k_t, so reading with q_t = k_t returns v_t (DeltaNet, Gated DeltaNet, KDA);
 *   3. a brute force by explicit d x d matrices, W <- W D (I - beta k k^T) +
 *      beta v k^T and o = W q (Sec. 2.3-2.5, Eqs. 14-20), at d = 4, T = 8;
 *   4. the mode reductions: KDA with the same log-decay on every key channel is
 *      Gated DeltaNet, and Gated DeltaNet with zero log-decay is DeltaNet;
 *   5. state passing: running T1 tokens, then T2 tokens from the returned state,
 *      equals running T1 + T2 tokens (the state travels through fp32, as the
 *      oracle's interface takes it, hence a 1e-6 tolerance on that check).
 * Prints one line per check and exits non-zero if any fails.
 */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

int ldn_oracle_fwd(const float *q, const float *k, const float *v, const float *beta, const float *gate,
                   const float *S0, double *out, double *S_final, int B, int T, int H, int dk, int dv, int mode,
                   int nthreads, int *threads_used);

enum { DN = 0, GDN = 1, KDA = 2 };
enum { D = 4, TT = 8 };

static int failures = 0;

static void report(const char *name, double err, double tol)
{
    const int ok = err <= tol;
    printf("%s %s (max err %.3g, tol %.3g)\n", ok ? "ok  " : "FAIL", name, err, tol);
    if (!ok) ++failures;
}

/* A small deterministic generator (xorshift64*) for the random cases. */
static unsigned long long rng_state = 0x9E3779B97F4A7C15ull;
static double urand(void)
{
    rng_state ^= rng_state >> 12;
    rng_state ^= rng_state << 25;
    rng_state ^= rng_state >> 27;
    return (double)((rng_state * 2685821657736338717ull) >> 11) * (1.0 / 9007199254740992.0);
}
static float srand1(void) { return (float)(2.0 * urand() - 1.0); }

static void check_worked_example(void)
{
    /* dk = 2, dv = 1; H = W^T holds the prediction for e0 (2) and for e1 (7). */
    const float S0[2] = {2.0f, 7.0f};
    const float k[2] = {1.0f, 0.0f}, v[1] = {5.0f}, beta[1] = {0.5f};
    const float q_key[2] = {1.0f, 0.0f}, q_orth[2] = {0.0f, 1.0f};
    double o = 0.0, sf[2] = {0.0, 0.0}, o2 = 0.0;
    int rc = ldn_oracle_fwd(q_key, k, v, beta, NULL, S0, &o, sf, 1, 1, 1, 2, 1, DN, 1, NULL);
    rc |= ldn_oracle_fwd(q_orth, k, v, beta, NULL, S0, &o2, NULL, 1, 1, 1, 2, 1, DN, 1, NULL);
    double err = rc ? 1.0 : fabs(o - 3.5);
    err = fmax(err, fabs(sf[0] - 3.5));
    err = fmax(err, fabs(o2 - 7.0));
    err = fmax(err, fabs(sf[1] - 7.0));
    report("worked example: prediction 2 -> 3.5 for target 5, beta 0.5", err, 0.0);
}

/* Random inputs for one (b, h) at d = 4, T = 8. */
typedef struct {
    float q[TT * D], k[TT * D], v[TT * D], beta[TT], g_gdn[TT], g_kda[TT * D], S0[D * D];
} case_t;

static void make_case(case_t *c, int axis_keys, int unit_beta)
{
    for (int t = 0; t < TT; ++t) {
        double n = 0.0;
        for (int i = 0; i < D; ++i) {
            c->q[t * D + i] = srand1();
            c->k[t * D + i] = srand1();
            c->v[t * D + i] = srand1();
            c->g_kda[t * D + i] = (float)(-0.3 * urand());
            n += (double)c->k[t * D + i] * c->k[t * D + i];
        }
        if (axis_keys) {
            const int a = (int)(urand() * D) % D;
            for (int i = 0; i < D; ++i) c->k[t * D + i] = i == a ? 1.0f : 0.0f;
        } else {
            for (int i = 0; i < D; ++i) c->k[t * D + i] = (float)(c->k[t * D + i] / sqrt(n));
        }
        c->beta[t] = unit_beta ? 1.0f : (float)urand();
        c->g_gdn[t] = (float)(-0.3 * urand());
    }
    for (int i = 0; i < D * D; ++i) c->S0[i] = (float)(0.5 * srand1());
}

static const float *gate_of(const case_t *c, int mode)
{
    return mode == GDN ? c->g_gdn : (mode == KDA ? c->g_kda : NULL);
}

static void check_exact_write(void)
{
    for (int mode = DN; mode <= KDA; ++mode) {
        case_t c;
        make_case(&c, 1, 1);
        double out[TT * D];
        const int rc = ldn_oracle_fwd(c.k, c.k, c.v, c.beta, gate_of(&c, mode), c.S0, out, NULL, 1, TT, 1, D, D,
                                      mode, 1, NULL);   /* read with q_t = k_t */
        double err = rc ? 1.0 : 0.0;
        for (int i = 0; i < TT * D; ++i) err = fmax(err, fabs(out[i] - (double)c.v[i]));
        char name[96];
        snprintf(name, sizeof name, "exact write at beta = 1, unit keys, mode %d", mode);
        report(name, err, 1e-13);
    }
}

/* W (dv x dk) <- W D (I - beta k k^T) + beta v k^T with every matrix formed explicitly. */
static void brute_force(const case_t *c, int mode, double *out, double *Wt_final)
{
    double W[D][D], M[D][D], N[D][D];
    for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j) W[i][j] = (double)c->S0[j * D + i];   /* S0 holds W^T */
    for (int t = 0; t < TT; ++t) {
        const float *k = c->k + t * D, *v = c->v + t * D, *q = c->q + t * D;
        const double b = c->beta[t];
        double Dm[D][D] = {{0}};
        for (int i = 0; i < D; ++i)
            Dm[i][i] = mode == DN ? 1.0 : exp(mode == GDN ? (double)c->g_gdn[t] : (double)c->g_kda[t * D + i]);
        for (int i = 0; i < D; ++i)           /* M = D (I - beta k k^T) */
            for (int j = 0; j < D; ++j) {
                double s = 0.0;
                for (int l = 0; l < D; ++l) s += Dm[i][l] * ((l == j ? 1.0 : 0.0) - b * (double)k[l] * (double)k[j]);
                M[i][j] = s;
            }
        for (int i = 0; i < D; ++i)           /* N = W M + beta v k^T */
            for (int j = 0; j < D; ++j) {
                double s = 0.0;
                for (int l = 0; l < D; ++l) s += W[i][l] * M[l][j];
                N[i][j] = s + b * (double)v[i] * (double)k[j];
            }
        memcpy(W, N, sizeof W);
        for (int i = 0; i < D; ++i) {         /* o = W q */
            double s = 0.0;
            for (int j = 0; j < D; ++j) s += W[i][j] * (double)q[j];
            out[t * D + i] = s;
        }
    }
    for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j) Wt_final[j * D + i] = W[i][j];
}

static double max_rel(const double *a, const double *b, int n)
{
    double m = 0.0, r = 0.0;
    for (int i = 0; i < n; ++i) {
        m = fmax(m, fabs(a[i] - b[i]));
        r = fmax(r, fabs(b[i]));
    }
    return r > 0.0 ? m / r : m;
}

static void check_brute_force(void)
{
    for (int mode = DN; mode <= KDA; ++mode) {
        case_t c;
        make_case(&c, 0, 0);
        double out[TT * D], sf[D * D], bo[TT * D], bs[D * D];
        const int rc = ldn_oracle_fwd(c.q, c.k, c.v, c.beta, gate_of(&c, mode), c.S0, out, sf, 1, TT, 1, D, D,
                                      mode, 1, NULL);
        brute_force(&c, mode, bo, bs);
        const double err = rc ? 1.0 : fmax(max_rel(out, bo, TT * D), max_rel(sf, bs, D * D));
        char name[96];
        snprintf(name, sizeof name, "brute force by explicit 4 x 4 matrices, mode %d", mode);
        report(name, err, 1e-12);
    }
}

static void check_mode_reductions(void)
{
    case_t c;
    make_case(&c, 0, 0);
    float g_same[TT * D], g_zero[TT];
    for (int t = 0; t < TT; ++t) {
        g_zero[t] = 0.0f;
        for (int i = 0; i < D; ++i) g_same[t * D + i] = c.g_gdn[t];
    }
    double o1[TT * D], s1[D * D], o2[TT * D], s2[D * D];
    int rc = ldn_oracle_fwd(c.q, c.k, c.v, c.beta, g_same, c.S0, o1, s1, 1, TT, 1, D, D, KDA, 1, NULL);
    rc |= ldn_oracle_fwd(c.q, c.k, c.v, c.beta, c.g_gdn, c.S0, o2, s2, 1, TT, 1, D, D, GDN, 1, NULL);
    report("KDA with one log-decay on every channel is Gated DeltaNet",
           rc ? 1.0 : fmax(max_rel(o1, o2, TT * D), max_rel(s1, s2, D * D)), 1e-13);
    rc = ldn_oracle_fwd(c.q, c.k, c.v, c.beta, g_zero, c.S0, o1, s1, 1, TT, 1, D, D, GDN, 1, NULL);
    rc |= ldn_oracle_fwd(c.q, c.k, c.v, c.beta, NULL, c.S0, o2, s2, 1, TT, 1, D, D, DN, 1, NULL);
    report("Gated DeltaNet with zero log-decay is DeltaNet",
           rc ? 1.0 : fmax(max_rel(o1, o2, TT * D), max_rel(s1, s2, D * D)), 0.0);
}

static void check_state_passing(void)
{
    for (int mode = DN; mode <= KDA; ++mode) {
        case_t c;
        make_case(&c, 0, 0);
        const int T1 = 3, T2 = TT - T1;
        const float *g = gate_of(&c, mode);
        const int gw = mode == KDA ? D : 1;
        double oall[TT * D], sall[D * D], o1[TT * D], s1[D * D], o2[TT * D], s2[D * D];
        float mid[D * D];
        int rc = ldn_oracle_fwd(c.q, c.k, c.v, c.beta, g, c.S0, oall, sall, 1, TT, 1, D, D, mode, 1, NULL);
        rc |= ldn_oracle_fwd(c.q, c.k, c.v, c.beta, g, c.S0, o1, s1, 1, T1, 1, D, D, mode, 1, NULL);
        for (int i = 0; i < D * D; ++i) mid[i] = (float)s1[i];
        rc |= ldn_oracle_fwd(c.q + T1 * D, c.k + T1 * D, c.v + T1 * D, c.beta + T1, g ? g + T1 * gw : NULL, mid,
                             o2, s2, 1, T2, 1, D, D, mode, 1, NULL);
        double err = rc ? 1.0 : fmax(max_rel(o1, oall, T1 * D), 0.0);
        err = fmax(err, max_rel(o2, oall + T1 * D, T2 * D));
        err = fmax(err, max_rel(s2, sall, D * D));
        char name[96];
        snprintf(name, sizeof name, "state passing T = 3 + 5 equals T = 8, mode %d", mode);
        report(name, err, 1e-6);
    }
}

int main(void)
{
    check_worked_example();
    check_exact_write();
    check_brute_force();
    check_mode_reductions();
    check_state_passing();
    printf("%d failure(s)\n", failures);
    return failures ? 1 : 0;
}
