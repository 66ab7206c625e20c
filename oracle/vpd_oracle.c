/*
 * vpd_oracle.c -- plain, slow, double-precision CPU oracle for the per-token
 * softmax divergences over a language-model vocabulary: the generalized
 * Jensen-Shannon divergence JSD_beta, forward/reverse KL, entropy and selected
 * (top-k) log-probabilities, each with its closed-form gradient.
 *
 * TEST INFRASTRUCTURE ONLY. The test suite, the smoke check and the benchmark's
 * CPU-baseline leg are the only code allowed to load this library. It shares
 * no code, header, table or helper with the GPU library, and neither links the
 * other.
 *
 * Sources (web pages; cited by short name below):
 *   [JSD page]  DeepSpeed pull request #8958, "[VocabTP] Add vocabulary-parallel
 *               generalized JSD with Triton kernels".
 *   [ops page]  DeepSpeed pull request #8791, "Add vocabulary-parallel logprobs,
 *               entropy and KL ops".
 *
 * Every function works one token row at a time, over the full vocabulary, in
 * the order of the steps below (no blocking, no fusion):
 *   1. The caller upcasts the logits exactly to double. Built with
 *      VPD_ORACLE_LONG_DOUBLE, every step below works in long double instead
 *      (the same steps and terms; only the rounding of the intermediates
 *      changes) and the outputs are rounded once to double.
 *   2. A row holding NaN or +inf is outside the contract; it is given a NaN
 *      output and an all-zero gradient (a reading: the pages are silent).
 *   3. Row statistics in two naive passes: the support S = {j : x_j > -inf},
 *      m = max_S x_j, Z = sum_S exp(x_j - m), L = ln Z. The max and the
 *      log-sum-exp stay separate ([ops page], "How": a large common offset
 *      must not cost precision), and ln p_j = (x_j - m) - L.
 *   4. The per-token value.
 *   5. The closed-form gradient, scaled by the upstream gradient g.
 *   6. Special values: a fully -inf row has no distribution, gives NaN and an
 *      exactly zero gradient ([ops page], "How" and the review thread "Prevent
 *      NaN gradients from fully masked padding rows"); a row whose KL is +inf
 *      (the target has mass on a token the other side masks, decided by logit
 *      finiteness, [ops page], "Tests") also gets a zero gradient.
 *
 * Sums over the vocabulary are plain left-to-right sums with Neumaier
 * compensation; they change only the rounding, not the order of the terms.
 * Natural logarithms (nats) throughout.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

/* ------------------------------------------------------------------------- */
/* Working precision: double, or with VPD_ORACLE_LONG_DOUBLE defined the       */
/* host's long double (80-bit extended on x86-64, 128-bit on AArch64). Inputs  */
/* and outputs stay double arrays; the values are upcast exactly on entry and  */
/* every intermediate is carried in the working precision.                    */
/* ------------------------------------------------------------------------- */
#ifdef VPD_ORACLE_LONG_DOUBLE
typedef long double real;
#define REXP expl
#define RLOG logl
#define RLOG1P log1pl
#define RFABS fabsl
#else
typedef double real;
#define REXP exp
#define RLOG log
#define RLOG1P log1p
#define RFABS fabs
#endif

/* ------------------------------------------------------------------------- */
/* Compensated running sum (Neumaier).                                        */
/* ------------------------------------------------------------------------- */
typedef struct {
    real sum;
    real comp;
} csum;

static void csum_add(csum *a, real v)
{
    real t = a->sum + v;
    if (RFABS(a->sum) >= RFABS(v))
        a->comp += (a->sum - t) + v;
    else
        a->comp += (v - t) + a->sum;
    a->sum = t;
}

static real csum_value(const csum *a) { return a->sum + a->comp; }

/* ------------------------------------------------------------------------- */
/* Step 2 and 3: row statistics.                                              */
/* ------------------------------------------------------------------------- */
typedef struct {
    int bad;      /* the row holds NaN or +inf (step 2)              */
    int empty;    /* the support is empty: every entry is -inf        */
    real m;       /* max over the support                             */
    real z;       /* sum over the support of exp(x_j - m)             */
    real lse;     /* ln z                                             */
} row_stats;

static row_stats stats_of(int64_t V, const double *x)
{
    row_stats r;
    r.bad = 0;
    r.empty = 1;
    r.m = -INFINITY;
    r.z = 0.0;
    r.lse = -INFINITY;
    /* pass 1: validity and the max over the support */
    for (int64_t j = 0; j < V; ++j) {
        real v = x[j];
        if (isnan(v) || v == INFINITY) {
            r.bad = 1;
            continue;
        }
        if (v == -INFINITY)
            continue;
        r.empty = 0;
        if (v > r.m)
            r.m = v;
    }
    if (r.bad || r.empty)
        return r;
    /* pass 2: the sum of exponentials relative to the max */
    csum z = {0.0, 0.0};
    for (int64_t j = 0; j < V; ++j) {
        real v = x[j];
        if (v == -INFINITY)
            continue;
        csum_add(&z, REXP(v - r.m));
    }
    r.z = csum_value(&z);
    r.lse = RLOG(r.z);
    return r;
}

/* ln p_j for an entry on the support */
static real log_prob(const row_stats *r, real x) { return (x - r->m) - r->lse; }

/* Public: per-row statistics (m, ln Z). Returns 1 for a NaN/+inf row, 2 for a
 * fully -inf row, 0 otherwise. */
int vpd_oracle_row_stats(int64_t V, const double *x, double *m, double *lse)
{
    row_stats r = stats_of(V, x);
    *m = r.m;
    *lse = r.lse;
    if (r.bad)
        return 1;
    if (r.empty)
        return 2;
    return 0;
}

/* Public: statistics merged over ordered vocabulary segments, the way
 * vocabulary shards are merged by a MAX all-reduce of the per-shard max and a
 * SUM all-reduce of the per-shard sum-exp ([ops page], "How"). A segment with
 * no finite entry (including an empty one) contributes (-inf, 0) ([ops page],
 * review thread "Reject unsupported empty shards consistently across TP
 * ranks"). Used only to check that the merge equals the full-row statistics.
 * Returns 1 if a width is negative or the widths do not sum to V. */
int vpd_oracle_segment_stats(int64_t V, const double *x, int count, const int64_t *widths,
                             double *m_out, double *z_out)
{
    int64_t total = 0;
    for (int k = 0; k < count; ++k) {
        if (widths[k] < 0)
            return 1;
        total += widths[k];
    }
    if (total != V)
        return 1;
    /* each segment on its own: (m_k, z_k) with z_k relative to m_k */
    real m = -INFINITY;
    int64_t off = 0;
    for (int k = 0; k < count; ++k) {
        row_stats r = stats_of(widths[k], x + off);
        if (!r.empty && r.m > m)
            m = r.m;
        off += widths[k];
    }
    csum z = {0.0, 0.0};
    off = 0;
    for (int k = 0; k < count; ++k) {
        row_stats r = stats_of(widths[k], x + off);
        if (!r.empty)
            csum_add(&z, r.z * REXP(r.m - m));
        off += widths[k];
    }
    *m_out = m;
    *z_out = csum_value(&z);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Helpers for the gradient outputs.                                          */
/* ------------------------------------------------------------------------- */
static void zero_row(double *d, int64_t V)
{
    if (!d)
        return;
    for (int64_t j = 0; j < V; ++j)
        d[j] = 0.0;
}

/* ln(a_w * e^{la} + b_w * e^{lb}) for log-weights lwa = ln a_w, lwb = ln b_w;
 * either log-argument may be -inf (the other then decides). */
static real log_mix(real lwa, real la, real lwb, real lb)
{
    real u = lwa + la;
    real v = lwb + lb;
    if (u == -INFINITY)
        return v;
    if (v == -INFINITY)
        return u;
    real hi = u > v ? u : v;
    real lo = u > v ? v : u;
    return hi + RLOG1P(REXP(lo - hi));
}

/* ------------------------------------------------------------------------- */
/* KL between two token distributions of one row.                             */
/*   KL(P_a || P_b) = sum_{j in S_a} a_j (ln a_j - ln b_j)                    */
/* +inf when some j has a_j > -inf logit but b_j = -inf logit ([ops page],     */
/* "Tests": decided by finiteness, even if the mass underflows in fp32).       */
/* Gradient ([ops page], "How": closed form, local):                           */
/*   d/d(logit_a)_j = g * a_j (ln a_j - ln b_j - KL)                           */
/*   d/d(logit_b)_j = g * (b_j - a_j)                                          */
/* ------------------------------------------------------------------------- */
static real kl_row(int64_t V, const double *xa, const double *xb, real g, double *da,
                     double *db)
{
    row_stats ra = stats_of(V, xa);
    row_stats rb = stats_of(V, xb);
    if (ra.bad || rb.bad || ra.empty || rb.empty) {
        zero_row(da, V);
        zero_row(db, V);
        return NAN;
    }
    for (int64_t j = 0; j < V; ++j) {
        if (xa[j] != -INFINITY && xb[j] == -INFINITY) {
            zero_row(da, V);
            zero_row(db, V);
            return INFINITY;
        }
    }
    csum kl = {0.0, 0.0};
    for (int64_t j = 0; j < V; ++j) {
        if (xa[j] == -INFINITY)
            continue;
        real la = log_prob(&ra, xa[j]);
        real lb = log_prob(&rb, xb[j]);
        csum_add(&kl, REXP(la) * (la - lb));
    }
    real value = csum_value(&kl);
    for (int64_t j = 0; j < V; ++j) {
        real a = xa[j] == -INFINITY ? 0.0 : REXP(log_prob(&ra, xa[j]));
        real b = xb[j] == -INFINITY ? 0.0 : REXP(log_prob(&rb, xb[j]));
        if (da) {
            if (xa[j] == -INFINITY)
                da[j] = 0.0;
            else
                da[j] = g * a * (log_prob(&ra, xa[j]) - log_prob(&rb, xb[j]) - value);
        }
        if (db)
            db[j] = g * (b - a);
    }
    return value;
}

/* ------------------------------------------------------------------------- */
/* Generalized JSD of one row ([JSD page], "Motivation" and "Changes").        */
/*   p = softmax(s) (student), q = softmax(t) (teacher),                      */
/*   M = (1 - beta) p + beta q,                                                */
/*   JSD_beta = beta * KL(q || M) + (1 - beta) * KL(p || M)                    */
/* beta = 0 is the explicit forward-KL branch KL(q || p), beta = 1 the explicit */
/* reverse-KL branch KL(p || q); they are branches, not limits ([JSD page],    */
/* "Changes").                                                                  */
/* Interior gradient, with A = KL(q || M) and B = KL(p || M):                  */
/*   dS_j = g (1 - beta) p_j (ln p_j - ln M_j - B)                             */
/*   dT_j = g beta       q_j (ln q_j - ln M_j - A)                             */
/* ------------------------------------------------------------------------- */
static real jsd_row(int64_t V, const double *s, const double *t, real beta, real g,
                      double *ds, double *dt, real *a_out, real *b_out)
{
    *a_out = NAN;
    *b_out = NAN;
    if (beta == 0.0) /* forward KL: target is the teacher */
        return kl_row(V, t, s, g, dt, ds);
    if (beta == 1.0) /* reverse KL: target is the student */
        return kl_row(V, s, t, g, ds, dt);

    row_stats rs = stats_of(V, s);
    row_stats rt = stats_of(V, t);
    if (rs.bad || rt.bad || rs.empty || rt.empty) {
        zero_row(ds, V);
        zero_row(dt, V);
        return NAN;
    }
    const real lw_s = RLOG(1.0 - beta); /* log-weight of p in M */
    const real lw_t = RLOG(beta);       /* log-weight of q in M */

    /* the two KL-to-mixture expectations, reduced together */
    csum A = {0.0, 0.0};
    csum B = {0.0, 0.0};
    for (int64_t j = 0; j < V; ++j) {
        int in_s = s[j] != -INFINITY;
        int in_t = t[j] != -INFINITY;
        if (!in_s && !in_t)
            continue;
        real lp = in_s ? log_prob(&rs, s[j]) : -INFINITY;
        real lq = in_t ? log_prob(&rt, t[j]) : -INFINITY;
        real lm = log_mix(lw_s, lp, lw_t, lq);
        if (in_t)
            csum_add(&A, REXP(lq) * (lq - lm));
        if (in_s)
            csum_add(&B, REXP(lp) * (lp - lm));
    }
    real a = csum_value(&A);
    real b = csum_value(&B);
    *a_out = a;
    *b_out = b;
    real value = beta * a + (1.0 - beta) * b;

    for (int64_t j = 0; j < V; ++j) {
        int in_s = s[j] != -INFINITY;
        int in_t = t[j] != -INFINITY;
        if (!in_s && !in_t) {
            if (ds)
                ds[j] = 0.0;
            if (dt)
                dt[j] = 0.0;
            continue;
        }
        real lp = in_s ? log_prob(&rs, s[j]) : -INFINITY;
        real lq = in_t ? log_prob(&rt, t[j]) : -INFINITY;
        real lm = log_mix(lw_s, lp, lw_t, lq);
        if (ds)
            ds[j] = in_s ? g * (1.0 - beta) * REXP(lp) * (lp - lm - b) : 0.0;
        if (dt)
            dt[j] = in_t ? g * beta * REXP(lq) * (lq - lm - a) : 0.0;
    }
    return value;
}

/* ------------------------------------------------------------------------- */
/* Entropy of one row ([ops page], "What"):                                    */
/*   H = - sum_{j in S} p_j ln p_j,   dX_j = -g p_j (ln p_j + H)               */
/* ------------------------------------------------------------------------- */
static real entropy_row(int64_t V, const double *x, real g, double *dx)
{
    row_stats r = stats_of(V, x);
    if (r.bad || r.empty) {
        zero_row(dx, V);
        return NAN;
    }
    csum h = {0.0, 0.0};
    for (int64_t j = 0; j < V; ++j) {
        if (x[j] == -INFINITY)
            continue;
        real lp = log_prob(&r, x[j]);
        csum_add(&h, -REXP(lp) * lp);
    }
    real value = csum_value(&h);
    if (dx) {
        for (int64_t j = 0; j < V; ++j) {
            if (x[j] == -INFINITY) {
                dx[j] = 0.0;
                continue;
            }
            real lp = log_prob(&r, x[j]);
            dx[j] = -g * REXP(lp) * (lp + value);
        }
    }
    return value;
}

/* ------------------------------------------------------------------------- */
/* Public batched entry points. Arrays are dense row-major [N, V] doubles;     */
/* g is [N] (NULL means 1 for every row); gradient pointers may be NULL.       */
/* ------------------------------------------------------------------------- */
void vpd_oracle_jsd(int64_t N, int64_t V, const double *s, const double *t, double beta,
                    const double *g, double *loss, double *kl_tm, double *kl_sm, double *ds,
                    double *dt)
{
    for (int64_t r = 0; r < N; ++r) {
        real a, b;
        loss[r] = jsd_row(V, s + r * V, t + r * V, beta, g ? g[r] : 1.0, ds ? ds + r * V : NULL,
                          dt ? dt + r * V : NULL, &a, &b);
        if (kl_tm)
            kl_tm[r] = a;
        if (kl_sm)
            kl_sm[r] = b;
    }
}

/* reverse = 0: KL(P_t || P_s) (forward KL, teacher is the target);
 * reverse = 1: KL(P_s || P_t) ([ops page], "What"). */
void vpd_oracle_kl(int64_t N, int64_t V, const double *s, const double *t, int reverse,
                   const double *g, double *loss, double *ds, double *dt)
{
    for (int64_t r = 0; r < N; ++r) {
        real gr = g ? g[r] : 1.0;
        double *dsr = ds ? ds + r * V : NULL;
        double *dtr = dt ? dt + r * V : NULL;
        if (reverse)
            loss[r] = kl_row(V, s + r * V, t + r * V, gr, dsr, dtr);
        else
            loss[r] = kl_row(V, t + r * V, s + r * V, gr, dtr, dsr);
    }
}

void vpd_oracle_entropy(int64_t N, int64_t V, const double *x, const double *g, double *out,
                        double *dx)
{
    for (int64_t r = 0; r < N; ++r)
        out[r] = entropy_row(V, x + r * V, g ? g[r] : 1.0, dx ? dx + r * V : NULL);
}

/* Selected log-probabilities ([ops page], "What"): out[r,k] = ln p_{i_rk};
 * a position equal to ignore_index returns 0 and takes no gradient; an index
 * outside [0, V) is an error (counted in the return value; its output is NaN).
 * A selected token with a -inf logit has log-prob -inf. Gradient over the
 * valid positions k whose output is finite:
 *   dX_j = sum_k g_rk [j == i_rk] - p_j sum_k g_rk.
 * g is [N, K] (NULL means 1). */
int64_t vpd_oracle_logprobs(int64_t N, int64_t V, const double *x, int64_t K, const int64_t *idx,
                            int64_t ignore_index, const double *g, double *out, double *dx)
{
    int64_t errors = 0;
    for (int64_t r = 0; r < N; ++r) {
        const double *xr = x + r * V;
        double *dxr = dx ? dx + r * V : NULL;
        row_stats st = stats_of(V, xr);
        int undefined = st.bad || st.empty;
        csum gsum = {0.0, 0.0};
        zero_row(dxr, V);
        for (int64_t k = 0; k < K; ++k) {
            int64_t i = idx[r * K + k];
            real gk = g ? g[r * K + k] : 1.0;
            real v;
            if (i == ignore_index) {
                out[r * K + k] = 0.0;
                continue;
            }
            if (i < 0 || i >= V) {
                ++errors;
                out[r * K + k] = NAN;
                continue;
            }
            if (undefined)
                v = NAN;
            else if (xr[i] == -INFINITY)
                v = -INFINITY;
            else
                v = log_prob(&st, xr[i]);
            out[r * K + k] = v;
            if (!isfinite(v))
                continue; /* a non-finite output takes no gradient */
            if (dxr)
                dxr[i] += gk;
            csum_add(&gsum, gk);
        }
        if (dxr && !undefined) {
            real gs = csum_value(&gsum);
            for (int64_t j = 0; j < V; ++j) {
                if (xr[j] == -INFINITY)
                    continue;
                dxr[j] -= REXP(log_prob(&st, xr[j])) * gs;
            }
        }
    }
    return errors;
}
