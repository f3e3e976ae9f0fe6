/*
 * fp64 CPU oracle for lossless speculative-sampling verification.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the verification computes.  It is compiled and called
 * only by the tests, by the smoke check and by the benchmark's CPU-baseline
 * leg; the library under speculative_decoding_verification_71_gb300/ never
 * links, loads or calls it, and the two share no source.
 *
 * What it computes (one sequence b at a time, all arithmetic in double):
 *   The verifier accepts or rejects each drafted token from the verifier's
 *   probability distribution, so that the rollout keeps the target policy's
 *   distribution ("Accelerating RL Post-Training Rollouts via
 *   System-Integrated Speculative Decoding", §2 core mechanism: rejection
 *   sampling).  It checks the drafts together and rewrites from the first
 *   wrong token ("Online Draft Co-Training for Speculative Decoding in
 *   Large-Scale, Long-Context RL Post-Training", the stenographer/proof-reader
 *   analogy).  The pages do not spell the rule out; the reading used is the
 *   standard speculative-sampling rule:
 *     p_i = softmax(z^t_i / T), q_i = softmax(z^d_i / T)
 *     accept draft i iff u_i < min(1, p_i(x_i) / q_i(x_i)); stop at the first
 *     rejection a;
 *     if a < k_b sample y from max(0, p_a - q_a) (normalised), else sample the
 *     bonus token y from p_{k_b};
 *     sampling is inverse CDF in ascending token id with the one sampling
 *     uniform s = u_{b,k}: y = min{x : s * S < C(x)}, C the running sum of
 *     the weights, S their total.
 *   q(x) = 0 for a drafted token gives r = +inf when p(x) > 0 and r = 0 when
 *   p(x) = 0.  T == 0 is greedy: accept iff x_i is the first argmax of p_i;
 *   the emitted token is the first argmax of the decided target row.
 *
 * Status per sequence: 0 ok, 2 draft length outside [0,k], 3 drafted token
 * outside [0,V), 4 NaN or +inf in a needed row or a needed row that is all
 * -inf.  A sequence with a nonzero status emits nothing (out_len 0, tokens
 * -1).  Bit 8 is set (status stays "ok") when the residual mass was exactly
 * zero and the sample was taken from p_a instead.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_BAD_DRAFT_LEN 2
#define ORC_BAD_TOKEN 3
#define ORC_NONFINITE 4
#define ORC_FLAG_ZERO_RESIDUAL 256

/* One logit as a double: fp32 widened, or bf16 bits placed in the top half
 * of an fp32 word and widened.  Both conversions are exact. */
static double logit_value(const void *base, int dtype, size_t idx)
{
    if (dtype == 0)
        return (double)((const float *)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static void load_row(const void *base, int dtype, size_t row, int V, double *out)
{
    size_t off = row * (size_t)V;
    for (int x = 0; x < V; ++x)
        out[x] = logit_value(base, dtype, off + (size_t)x);
}

/* A row may hold -inf (masked tokens) but no NaN or +inf, and not only -inf. */
static int row_is_valid(const double *z, int V)
{
    int finite_seen = 0;
    for (int x = 0; x < V; ++x) {
        if (isnan(z[x]) || z[x] == INFINITY)
            return 0;
        if (z[x] != -INFINITY)
            finite_seen = 1;
    }
    return finite_seen;
}

/* Row maximum m and L = log sum_x exp((z_x - m)/T), so that
 * log-sum-exp(z/T) = m/T + L and p(x) = exp((z_x - m)/T - L). */
static void row_stats(const double *z, int V, double T, double *m_out, double *L_out)
{
    double m = -INFINITY;
    for (int x = 0; x < V; ++x)
        if (z[x] > m)
            m = z[x];
    double s = 0.0;
    for (int x = 0; x < V; ++x)
        s += exp((z[x] - m) / T);
    *m_out = m;
    *L_out = log(s);
}

static double prob_of(double zx, double m, double L, double T)
{
    return exp((zx - m) / T - L);
}

static int first_argmax(const double *z, int V)
{
    int best = 0;
    for (int x = 1; x < V; ++x)
        if (z[x] > z[best])
            best = x;
    return best;
}

/* Inverse CDF over weights w[0..V): the smallest x with s*S < C(x); if
 * rounding leaves no such x, the last x with w(x) > 0.  Also returns the
 * distance of s, in units of C/S, to the two boundaries of the chosen x. */
static int inverse_cdf(const double *w, int V, double S, double s, double *tie)
{
    double t = s * S, c = 0.0, c_prev = 0.0;
    int y = -1;
    for (int x = 0; x < V; ++x) {
        c_prev = c;
        c += w[x];
        if (t < c) {
            y = x;
            break;
        }
    }
    if (y < 0) {
        for (int x = V - 1; x >= 0; --x)
            if (w[x] > 0.0) {
                y = x;
                break;
            }
        c = 0.0;
        for (int x = 0; x <= y; ++x)
            c += w[x];
        c_prev = c - w[y];
    }
    double d0 = fabs(s - c_prev / S), d1 = fabs(s - c / S);
    *tie = d0 < d1 ? d0 : d1;
    return y;
}

/* The tokens a draw could give if the uniform moved by at most `band` (in
 * units of C/S): the smallest and the largest x with w(x) > 0 whose CDF
 * interval [C(x-1), C(x)] comes within band * S of s * S.  When s lies that
 * close to a boundary of the drawn token, any token in [lo, hi] is a valid
 * outcome of a computation whose CDF is off by less than band. */
static void cdf_window(const double *w, int V, double S, double s, double band, int *lo, int *hi)
{
    double t_lo = (s - band) * S, t_hi = (s + band) * S, c_prev = 0.0, c = 0.0;
    *lo = -1;
    *hi = -1;
    for (int x = 0; x < V; ++x) {
        c_prev = c;
        c += w[x];
        if (w[x] > 0.0 && c >= t_lo && c_prev <= t_hi) {
            if (*lo < 0)
                *lo = x;
            *hi = x;
        }
    }
}

/*
 * oracle_verify: see the file comment.  Shapes as in the library:
 *   target [B,k+1,V], draft [B,k,V] (dtype 0 = fp32, 1 = bf16 bits),
 *   tokens [B,k], draft_len [B], uniforms [B,k+1] (float32),
 *   out_tokens [B,k+1] (-1 padded), out_len [B].
 * Optional diagnostics (any may be NULL):
 *   lse_t [B,k+1], lse_d [B,k]   log-sum-exp of z/T per needed row (NaN if
 *                                not needed or T == 0)
 *   p_x, q_x [B,k]               p_i(x_i), q_i(x_i)
 *   alpha [B,k]                  min(1, p_i(x_i)/q_i(x_i)) for every draft
 *                                (greedy: 1 if accepted else 0)
 *   resid_mass [B]               S of the sampled weights
 *   accept_tie [B]               min |u_i - alpha_i| over the tests that
 *                                decided a (1 if none)
 *   sample_tie [B]               distance of s to the chosen x's CDF bounds
 *   sample_lo, sample_hi [B]     the window of valid draws for a uniform off
 *                                by at most tie_band (see cdf_window); greedy:
 *                                both are the emitted token
 *   status [B]
 * nthreads <= 0 uses the OpenMP default.  Returns the number of sequences
 * with a nonzero status (flags excluded).
 */
int oracle_verify(int B, int k, int V, int dtype,
                  const void *target, const void *draft,
                  const int32_t *tokens, const int32_t *draft_len,
                  const float *uniforms, double T,
                  int32_t *out_tokens, int32_t *out_len,
                  double *lse_t, double *lse_d, double *p_x, double *q_x,
                  double *alpha, double *resid_mass, double *accept_tie,
                  double *sample_tie, double tie_band, int32_t *sample_lo,
                  int32_t *sample_hi, int32_t *status, int nthreads)
{
    int nerr = 0;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(+ : nerr)
#endif
    for (int b = 0; b < B; ++b) {
        double *zt = (double *)malloc(sizeof(double) * (size_t)V);
        double *zd = (double *)malloc(sizeof(double) * (size_t)V);
        double *w = (double *)malloc(sizeof(double) * (size_t)V);
        double *mt = (double *)malloc(sizeof(double) * (size_t)(k + 1) * 2);
        double *Lt = mt + (k + 1);
        double *md = (double *)malloc(sizeof(double) * (size_t)(k + 1) * 2);
        double *Ld = md + (k + 1);
        int *amax_t = (int *)malloc(sizeof(int) * (size_t)(k + 1));
        int st = ORC_OK;

        for (int j = 0; j <= k; ++j)
            out_tokens[(size_t)b * (k + 1) + j] = -1;
        out_len[b] = 0;
        for (int j = 0; j <= k; ++j) {
            if (lse_t) lse_t[(size_t)b * (k + 1) + j] = NAN;
            if (j < k) {
                if (lse_d) lse_d[(size_t)b * k + j] = NAN;
                if (p_x) p_x[(size_t)b * k + j] = NAN;
                if (q_x) q_x[(size_t)b * k + j] = NAN;
                if (alpha) alpha[(size_t)b * k + j] = NAN;
            }
        }
        if (resid_mass) resid_mass[b] = NAN;
        if (accept_tie) accept_tie[b] = 1.0;
        if (sample_tie) sample_tie[b] = 1.0;
        if (sample_lo) sample_lo[b] = -1;
        if (sample_hi) sample_hi[b] = -1;

        int kb = draft_len[b];
        if (kb < 0 || kb > k)
            st = ORC_BAD_DRAFT_LEN;
        for (int i = 0; st == ORC_OK && i < kb; ++i) {
            int x = tokens[(size_t)b * k + i];
            if (x < 0 || x >= V)
                st = ORC_BAD_TOKEN;
        }
        /* Row statistics of every needed row. */
        for (int i = 0; st == ORC_OK && i <= kb; ++i) {
            load_row(target, dtype, (size_t)b * (k + 1) + i, V, zt);
            if (!row_is_valid(zt, V)) {
                st = ORC_NONFINITE;
                break;
            }
            amax_t[i] = first_argmax(zt, V);
            if (T > 0.0) {
                row_stats(zt, V, T, &mt[i], &Lt[i]);
                if (lse_t) lse_t[(size_t)b * (k + 1) + i] = mt[i] / T + Lt[i];
            }
            if (i < kb) {
                load_row(draft, dtype, (size_t)b * k + i, V, zd);
                if (!row_is_valid(zd, V)) {
                    st = ORC_NONFINITE;
                    break;
                }
                if (T > 0.0) {
                    row_stats(zd, V, T, &md[i], &Ld[i]);
                    if (lse_d) lse_d[(size_t)b * k + i] = md[i] / T + Ld[i];
                }
            }
        }
        if (st != ORC_OK) {
            if (status) status[b] = st;
            nerr += 1;
            free(zt); free(zd); free(w); free(mt); free(md); free(amax_t);
            continue;
        }

        const float *u = uniforms + (size_t)b * (k + 1);
        int a = kb;
        double atie = 1.0;
        if (T > 0.0) {
            /* Acceptance test of every draft (diagnostics), first rejection a. */
            int decided = 0;
            for (int i = 0; i < kb; ++i) {
                int x = tokens[(size_t)b * k + i];
                double zt_x = logit_value(target, dtype, ((size_t)b * (k + 1) + i) * (size_t)V + x);
                double zd_x = logit_value(draft, dtype, ((size_t)b * k + i) * (size_t)V + x);
                double p = prob_of(zt_x, mt[i], Lt[i], T);
                double q = prob_of(zd_x, md[i], Ld[i], T);
                double r = (q == 0.0) ? (p > 0.0 ? INFINITY : 0.0) : p / q;
                double al = r < 1.0 ? r : 1.0;
                if (p_x) p_x[(size_t)b * k + i] = p;
                if (q_x) q_x[(size_t)b * k + i] = q;
                if (alpha) alpha[(size_t)b * k + i] = al;
                if (!decided) {
                    double d = fabs((double)u[i] - al);
                    if (d < atie) atie = d;
                    if (!((double)u[i] < al)) {
                        a = i;
                        decided = 1;
                    }
                }
            }
            /* Weights of the final draw: residual at a, or bonus row k_b. */
            double S = 0.0;
            int flags = 0;
            load_row(target, dtype, (size_t)b * (k + 1) + a, V, zt);
            if (a < kb) {
                load_row(draft, dtype, (size_t)b * k + a, V, zd);
                for (int x = 0; x < V; ++x) {
                    double d = prob_of(zt[x], mt[a], Lt[a], T) - prob_of(zd[x], md[a], Ld[a], T);
                    w[x] = d > 0.0 ? d : 0.0;
                }
            } else {
                for (int x = 0; x < V; ++x)
                    w[x] = prob_of(zt[x], mt[a], Lt[a], T);
            }
            for (int x = 0; x < V; ++x)
                S += w[x];
            if (S == 0.0) {
                flags |= ORC_FLAG_ZERO_RESIDUAL;
                for (int x = 0; x < V; ++x)
                    w[x] = prob_of(zt[x], mt[a], Lt[a], T);
                S = 0.0;
                for (int x = 0; x < V; ++x)
                    S += w[x];
            }
            double stie = 1.0;
            int y = inverse_cdf(w, V, S, (double)u[k], &stie);
            int wlo, whi;
            cdf_window(w, V, S, (double)u[k], tie_band, &wlo, &whi);
            if (resid_mass) resid_mass[b] = S;
            if (sample_tie) sample_tie[b] = stie;
            if (sample_lo) sample_lo[b] = wlo;
            if (sample_hi) sample_hi[b] = whi;
            if (accept_tie) accept_tie[b] = atie;
            for (int i = 0; i < a; ++i)
                out_tokens[(size_t)b * (k + 1) + i] = tokens[(size_t)b * k + i];
            out_tokens[(size_t)b * (k + 1) + a] = y;
            out_len[b] = a + 1;
            if (status) status[b] = flags;
        } else {
            /* Greedy: accept iff the draft is the first argmax of p_i. */
            for (int i = 0; i < kb; ++i) {
                int x = tokens[(size_t)b * k + i];
                int ok = (x == amax_t[i]);
                if (alpha) alpha[(size_t)b * k + i] = ok ? 1.0 : 0.0;
                if (!ok && a == kb)
                    a = i;
            }
            for (int i = 0; i < a; ++i)
                out_tokens[(size_t)b * (k + 1) + i] = tokens[(size_t)b * k + i];
            out_tokens[(size_t)b * (k + 1) + a] = amax_t[a];
            out_len[b] = a + 1;
            if (sample_lo) sample_lo[b] = amax_t[a];
            if (sample_hi) sample_hi[b] = amax_t[a];
            if (status) status[b] = ORC_OK;
        }
        free(zt); free(zd); free(w); free(mt); free(md); free(amax_t);
    }
    return nerr;
}

/* Row maximum and L (as in row_stats) of one row, for checking the
 * log-sum-exp against a library routine.  Returns m/T + L. */
double oracle_row_lse(int V, int dtype, const void *row, double T)
{
    double *z = (double *)calloc((size_t)V, sizeof(double));
    load_row(row, dtype, 0, V, z);
    double m, L;
    row_stats(z, V, T, &m, &L);
    free(z);
    return m / T + L;
}

/* p(x) = softmax(z/T)(x) for every x of one row. */
void oracle_row_probs(int V, int dtype, const void *row, double T, double *p)
{
    double *z = (double *)calloc((size_t)V, sizeof(double));
    load_row(row, dtype, 0, V, z);
    double m, L;
    row_stats(z, V, T, &m, &L);
    for (int x = 0; x < V; ++x)
        p[x] = prob_of(z[x], m, L, T);
    free(z);
}

/* Widening of one logit (exposed so that the exact bf16/fp32 conversion can
 * be checked against the framework's own conversion). */
double oracle_logit_value(const void *base, int dtype, long long idx)
{
    return logit_value(base, dtype, (size_t)idx);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Reward-weighted distillation loss of the draft model ("ReSpec: Towards
 * Optimizing Speculative Decoding in Reinforcement Learning Systems", Online
 * Learner, reward-weighted KD): each rollout b of t_len positions adds
 *   L_b = w_b * sum_t KL(pt_{b,t} || q_{b,t}),
 *   pt = softmax(z^t / T) (the updated target), q = softmax(z^d / T) (draft),
 *   KL(p || q) = sum_x p(x) (log p(x) - log q(x)),
 * where a term with p(x) = 0 is 0 and p(x) > 0 with q(x) = 0 makes KL = +inf.
 * The gradient with respect to the draft logits is
 *   dL_b / dz^d_{b,t}(x) = w_b (q(x) - pt(x)) / T.
 * w_b = w(r_b) is an input per rollout: the page weights the KL by a function
 * of the reward without fixing it.
 *
 * Per row, all in double: the row maximum and L of row_stats, then every
 * log-probability from them.  A row pair with NaN or +inf, or a row that is
 * all -inf, has status 4: its KL and gradient are NaN and so is its loss.
 * The loss sums the rows of a rollout in position order.
 * row_kl [n_seq * t_len], loss [n_seq], grad [n_seq * t_len * V] (may be
 * NULL), status [n_seq * t_len] (may be NULL).
 */
int oracle_kd(int n_seq, int t_len, int V, int dtype, const void *target, const void *draft,
              const double *weights, double T, double *row_kl, double *loss, double *grad,
              int *status, int nthreads)
{
    if (n_seq <= 0 || t_len <= 0 || V <= 0 || !(T > 0.0))
        return -1;
    const long long rows = (long long)n_seq * t_len;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#endif
    int bad_alloc = 0;
#pragma omp parallel reduction(| : bad_alloc)
    {
        double *zt = (double *)malloc(sizeof(double) * (size_t)V);
        double *zd = (double *)malloc(sizeof(double) * (size_t)V);
        if (!zt || !zd) {
            bad_alloc = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long long r = 0; r < rows; ++r) {
                const double w = weights[r / t_len];
                load_row(target, dtype, (size_t)r, V, zt);
                load_row(draft, dtype, (size_t)r, V, zd);
                int st = (row_is_valid(zt, V) && row_is_valid(zd, V)) ? ORC_OK : ORC_NONFINITE;
                if (status)
                    status[r] = st;
                if (st != ORC_OK) {
                    row_kl[r] = NAN;
                    if (grad)
                        for (int x = 0; x < V; ++x)
                            grad[(size_t)r * V + x] = NAN;
                    continue;
                }
                double mt, Lt, md, Ld;
                row_stats(zt, V, T, &mt, &Lt);
                row_stats(zd, V, T, &md, &Ld);
                double kl = 0.0;
                for (int x = 0; x < V; ++x) {
                    const double lp = (zt[x] - mt) / T - Lt;      /* log p(x) */
                    const double lq = (zd[x] - md) / T - Ld;      /* log q(x) */
                    const double p = exp(lp), q = exp(lq);
                    if (p > 0.0)
                        kl += p * (lp - lq);                     /* +inf when q(x) = 0 */
                    if (grad)
                        grad[(size_t)r * V + x] = w * (q - p) / T;
                }
                row_kl[r] = kl;
            }
        }
        free(zt);
        free(zd);
    }
    if (bad_alloc)
        return -2;
    for (int b = 0; b < n_seq; ++b) {
        double s = 0.0;
        for (int t = 0; t < t_len; ++t)
            s += row_kl[(size_t)b * t_len + t];
        loss[b] = weights[b] * s;
    }
    return 0;
}

/*
 * Acceptance-aware draft-length controller with the speculation toggle
 * ("EfficientRollout: System-Aware Self-Speculative Decoding for RL
 * Rollouts", abstract: a system-aware SD toggle with acceptance-aware
 * draft-length adaptation; "ReSpec: Towards Optimizing Speculative Decoding
 * in Reinforcement Learning Systems", Adaptive Server: a performance model
 * profiled offline per batch size picks the SD configuration for the
 * effective batch size, and the scheduler runs non-speculatively when the
 * batch is large).  The pages fix no formulas; the readings used:
 *
 *   observe: a round of sequence b with draft length k_b > 0 and emitted
 *     length out_len = a + 1 tested a + r drafts, r = 1 if a < k_b (the
 *     first rejection) else 0; drafts after a rejection are never tested.
 *     Decayed counts: A_b <- decay * A_b + a, N_b <- decay * N_b + (a + r).
 *   estimate: alpha_b = (A_b + alpha0 * w0) / (N_b + w0) (w0 prior
 *     pseudo-tests at rate alpha0); alpha0 when N_b + w0 = 0.  With decay 1
 *     and w0 = 0 this is the maximum-likelihood rate of the truncated
 *     geometric law of a.
 *   expected tokens of a round with draft length n at per-draft acceptance
 *     alpha: E_n(alpha) = sum_{j=0..n} alpha^j (the corrected or bonus token
 *     plus each accepted prefix).
 *   round time T(B, n): a table at profiled batch sizes B_0 < ... < B_m-1,
 *     linear in B between two of them, the end row outside.
 *   choose (mode 0, batch): n* = argmax_n sum_b E_n(alpha_b) / T(B, n) over
 *     n = 0..max_k, the smallest n on ties; every row gets n*; n* = 0 is
 *     speculation off.  (mode 1, per sequence): n_b = argmax_n
 *     E_n(alpha_b) / T(B, n).
 *
 * Row status: 0 used, 1 skipped (out_len 0: the verifier rejected the
 * sequence; or k_b = 0: nothing tested), 2 bad length (k_b outside
 * [0, max_k] or out_len outside [0, k_b + 1]), 5 bad id (outside
 * [0, n_slots) or repeated within the call).  Rows with status 2 or 5 leave
 * the state unchanged.
 */
#define ORC_CTRL_USED 0
#define ORC_CTRL_SKIPPED 1
#define ORC_CTRL_BAD_LEN 2
#define ORC_CTRL_BAD_ID 5

int oracle_ctrl_observe(int n_slots, double *A, double *N, int B, const int *seq_ids,
                        const int *draft_len, const int *out_len, int max_k, double decay,
                        int *row_status)
{
    for (int b = 0; b < B; ++b) {
        const int id = seq_ids[b];
        int repeated = 0;
        for (int c = 0; c < B; ++c)
            if (c != b && seq_ids[c] == id)
                repeated = 1;
        if (id < 0 || id >= n_slots || repeated) {
            row_status[b] = ORC_CTRL_BAD_ID;
            continue;
        }
        const int k = draft_len[b], len = out_len[b];
        if (k < 0 || k > max_k || len < 0 || len > k + 1) {
            row_status[b] = ORC_CTRL_BAD_LEN;
            continue;
        }
        if (len == 0 || k == 0) {
            row_status[b] = ORC_CTRL_SKIPPED;
            continue;
        }
        const int a = len - 1;
        const int r = (a < k) ? 1 : 0;
        A[id] = decay * A[id] + (double)a;
        N[id] = decay * N[id] + (double)(a + r);
        row_status[b] = ORC_CTRL_USED;
    }
    return 0;
}

double oracle_ctrl_alpha(double A, double N, double alpha0, double w0)
{
    const double den = N + w0;
    if (den == 0.0)
        return alpha0;
    return (A + alpha0 * w0) / den;
}

double oracle_ctrl_expected_tokens(double alpha, int n)
{
    double e = 0.0;
    for (int j = 0; j <= n; ++j)
        e += pow(alpha, (double)j);
    return e;
}

double oracle_ctrl_round_time(int n_points, const int *batch_sizes, const double *table,
                              int max_k, int B, int n)
{
    const int K1 = max_k + 1;
    if (B <= batch_sizes[0])
        return table[n];
    if (B >= batch_sizes[n_points - 1])
        return table[(size_t)(n_points - 1) * K1 + n];
    int j = 0;
    while (!(batch_sizes[j] <= B && B < batch_sizes[j + 1]))
        ++j;
    const double t0 = table[(size_t)j * K1 + n], t1 = table[(size_t)(j + 1) * K1 + n];
    const double f = (double)(B - batch_sizes[j]) / (double)(batch_sizes[j + 1] - batch_sizes[j]);
    return t0 + (t1 - t0) * f;
}

/* rates [max_k + 1] (may be NULL) receives, in batch mode, sum_b E_n / T(B, n);
 * margin (may be NULL) the relative gap between the best and the second-best
 * rate of the batch (mode 0) or of each row (mode 1, [B]).  Rows with a bad
 * id get 0 and status 5. */
int oracle_ctrl_choose(int n_slots, const double *A, const double *N, int B, const int *seq_ids,
                       int max_k, double alpha0, double w0, int mode, int n_points,
                       const int *batch_sizes, const double *table, int *next_len, int *choice,
                       double *rates, double *margin, int *row_status)
{
    const int K1 = max_k + 1;
    double T[32], R[32];
    if (K1 > 32)
        return -1;
    for (int n = 0; n < K1; ++n) {
        T[n] = oracle_ctrl_round_time(n_points, batch_sizes, table, max_k, B, n);
        R[n] = 0.0;
    }
    int best_all = 0;
    for (int b = 0; b < B; ++b) {
        const int id = seq_ids[b];
        if (id < 0 || id >= n_slots) {
            row_status[b] = ORC_CTRL_BAD_ID;
            next_len[b] = 0;
            if (mode == 1 && margin)
                margin[b] = INFINITY;
            continue;
        }
        row_status[b] = ORC_CTRL_USED;
        const double alpha = oracle_ctrl_alpha(A[id], N[id], alpha0, w0);
        if (mode == 0) {
            for (int n = 0; n < K1; ++n)
                R[n] += oracle_ctrl_expected_tokens(alpha, n);
            continue;
        }
        int best = 0;
        double top = -1.0, second = -1.0;
        for (int n = 0; n < K1; ++n) {
            const double rate = oracle_ctrl_expected_tokens(alpha, n) / T[n];
            if (rate > top) {
                second = top;
                top = rate;
                best = n;
            } else if (rate > second) {
                second = rate;
            }
        }
        next_len[b] = best;
        if (best > best_all)
            best_all = best;
        if (margin)
            margin[b] = (K1 > 1) ? (top - second) / top : INFINITY;
    }
    if (mode == 0) {
        int best = 0;
        double top = -1.0, second = -1.0;
        for (int n = 0; n < K1; ++n) {
            R[n] = R[n] / T[n];
            if (R[n] > top) {
                second = top;
                top = R[n];
                best = n;
            } else if (R[n] > second) {
                second = R[n];
            }
            if (rates)
                rates[n] = R[n];
        }
        for (int b = 0; b < B; ++b)
            if (row_status[b] == ORC_CTRL_USED)
                next_len[b] = best;
        best_all = best;
        if (margin)
            margin[0] = (K1 > 1 && top > 0.0) ? (top - second) / top : INFINITY;
    }
    if (choice)
        *choice = best_all;
    return 0;
}

/*
 * Tree verification ("ReSpec: Towards Optimizing Speculative Decoding in
 * Reinforcement Learning Systems", GAP 1: an SD configuration has a number of
 * rounds, a branching factor t and a draft length per round; the page gives
 * no verification rule for branching drafts).  Reading used: recursive
 * rejection sampling over a draft tree whose children at each node are
 * independent draws from the drafter's distribution q at that node, the
 * multi-candidate form of the rule of oracle_verify:
 *
 *   start at the root with r = p (the target distribution at the node);
 *   test the node's children in index order: child c with token x is
 *     accepted iff u_c < min(1, r(x) / q(x)) (r(x) > 0 = q(x) accepts);
 *     after a rejection w = max(0, r - q), S = sum_x w (index order), and
 *     r = w / S for the next child (S = 0: w = r, flagged);
 *   an accepted child emits its token and the walk continues at it;
 *   if every child was rejected, y is drawn from the last w, S; a node with
 *     no children draws the bonus token y from w = p, S = sum p;
 *   the draw is the inverse CDF of oracle_verify with the one sampling
 *     uniform s = u[b, 0].
 * A chain (one child per node) is exactly oracle_verify.  T == 0: the first
 * child whose token is the first argmax of the node's target row is accepted;
 * if none, or at a leaf, y is that argmax.
 *
 * Shapes: target, draft [B, M, V] (row j: after the path to node j; draft
 * row j is read only if node j has children), parents, tokens [B, M]
 * (node 0 is the root; 0 <= parents[j] < j for 1 <= j < n_nodes[b]),
 * n_nodes [B] in [1, M], uniforms [B, M] (column 0 samples, column j >= 1 is
 * child j's test).  Outputs: out_tokens [B, M] and out_nodes [B, M] (-1
 * padded; out_nodes holds the accepted nodes), out_len [B].  Optional (may
 * be NULL): alpha [B, M] (min(1, r(x)/q(x)) of each tested child, NaN if not
 * tested; greedy 1 or 0), final_w [B, V] (w / S of the draw), resid_mass [B]
 * (S of the draw), accept_tie [B] (min |u - alpha| over the tests made, 1 if
 * none), sample_tie [B], sample_lo / sample_hi [B] (the window of valid
 * draws for a uniform off by at most tie_band, as in oracle_verify), status
 * [B] (2 bad structure, 3 bad token, 4 a row
 * the walk reads is not finite or all -inf; flag 256: a zero residual).
 * Only the rows the walk reads are checked.
 */
int oracle_tree_verify(int B, int M, int V, int dtype, const void *target, const void *draft,
                       const int32_t *parents, const int32_t *tokens, const int32_t *n_nodes,
                       const float *uniforms, double T, int32_t *out_tokens, int32_t *out_nodes,
                       int32_t *out_len, double *alpha, double *final_w, double *resid_mass,
                       double *accept_tie, double *sample_tie, double tie_band, int32_t *sample_lo,
                       int32_t *sample_hi, int32_t *status, int nthreads)
{
    int nerr = 0;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(+ : nerr)
#endif
    for (int b = 0; b < B; ++b) {
        double *zt = (double *)malloc(sizeof(double) * (size_t)V);
        double *zd = (double *)malloc(sizeof(double) * (size_t)V);
        double *r = (double *)malloc(sizeof(double) * (size_t)V);
        double *q = (double *)malloc(sizeof(double) * (size_t)V);
        double *w = (double *)malloc(sizeof(double) * (size_t)V);
        const int32_t *par = parents + (size_t)b * M;
        const int32_t *tok = tokens + (size_t)b * M;
        const float *u = uniforms + (size_t)b * M;
        int32_t *ot = out_tokens + (size_t)b * M;
        int32_t *on = out_nodes + (size_t)b * M;
        for (int j = 0; j < M; ++j) {
            ot[j] = -1;
            on[j] = -1;
            if (alpha)
                alpha[(size_t)b * M + j] = NAN;
        }
        out_len[b] = 0;
        if (final_w)
            for (int x = 0; x < V; ++x)
                final_w[(size_t)b * V + x] = NAN;
        if (resid_mass) resid_mass[b] = NAN;
        if (accept_tie) accept_tie[b] = 1.0;
        if (sample_tie) sample_tie[b] = 1.0;
        if (sample_lo) sample_lo[b] = -1;
        if (sample_hi) sample_hi[b] = -1;

        int st = ORC_OK, flags = 0;
        const int n = n_nodes[b];
        if (n < 1 || n > M)
            st = ORC_BAD_DRAFT_LEN;
        for (int j = 1; st == ORC_OK && j < n; ++j)
            if (par[j] < 0 || par[j] >= j)
                st = ORC_BAD_DRAFT_LEN;
        for (int j = 1; st == ORC_OK && j < n; ++j)
            if (tok[j] < 0 || tok[j] >= V)
                st = ORC_BAD_TOKEN;

        int len = 0, cur = 0, y = -1;
        double atie = 1.0, stie = 1.0, S = 0.0;
        while (st == ORC_OK) {
            load_row(target, dtype, (size_t)b * M + cur, V, zt);
            if (!row_is_valid(zt, V)) {
                st = ORC_NONFINITE;
                break;
            }
            int has_children = 0;
            for (int c = cur + 1; c < n; ++c)
                if (par[c] == cur)
                    has_children = 1;
            if (has_children) {
                load_row(draft, dtype, (size_t)b * M + cur, V, zd);
                if (!row_is_valid(zd, V)) {
                    st = ORC_NONFINITE;
                    break;
                }
            }
            if (T == 0.0) {
                const int am = first_argmax(zt, V);
                int next = -1;
                for (int c = cur + 1; c < n && next < 0; ++c)
                    if (par[c] == cur) {
                        const int ok = (tok[c] == am);
                        if (alpha) alpha[(size_t)b * M + c] = ok ? 1.0 : 0.0;
                        if (ok) next = c;
                    }
                if (next < 0) {
                    y = am;
                    break;
                }
                on[len] = next;
                ot[len++] = tok[next];
                cur = next;
                continue;
            }
            double mt, Lt;
            row_stats(zt, V, T, &mt, &Lt);
            for (int x = 0; x < V; ++x)
                r[x] = prob_of(zt[x], mt, Lt, T);
            if (!has_children) {
                /* bonus token from p */
                S = 0.0;
                for (int x = 0; x < V; ++x) {
                    w[x] = r[x];
                    S += w[x];
                }
                break;
            }
            double md, Ld;
            row_stats(zd, V, T, &md, &Ld);
            for (int x = 0; x < V; ++x)
                q[x] = prob_of(zd[x], md, Ld, T);
            int next = -1;
            for (int c = cur + 1; c < n; ++c) {
                if (par[c] != cur)
                    continue;
                const int x = tok[c];
                const double ratio = (q[x] == 0.0) ? (r[x] > 0.0 ? INFINITY : 0.0) : r[x] / q[x];
                const double al = ratio < 1.0 ? ratio : 1.0;
                if (alpha) alpha[(size_t)b * M + c] = al;
                const double d = fabs((double)u[c] - al);
                if (d < atie) atie = d;
                if ((double)u[c] < al) {
                    next = c;
                    break;
                }
                S = 0.0;
                for (int xx = 0; xx < V; ++xx) {
                    const double v = r[xx] - q[xx];
                    w[xx] = v > 0.0 ? v : 0.0;
                    S += w[xx];
                }
                if (S == 0.0) {
                    flags |= ORC_FLAG_ZERO_RESIDUAL;
                    S = 0.0;
                    for (int xx = 0; xx < V; ++xx) {
                        w[xx] = r[xx];
                        S += w[xx];
                    }
                }
                for (int xx = 0; xx < V; ++xx)
                    r[xx] = w[xx] / S;
            }
            if (next < 0)
                break;                  /* every child rejected: draw from w, S */
            on[len] = next;
            ot[len++] = tok[next];
            cur = next;
        }
        int wlo = y, whi = y;
        if (st == ORC_OK && T > 0.0) {
            y = inverse_cdf(w, V, S, (double)u[0], &stie);
            cdf_window(w, V, S, (double)u[0], tie_band, &wlo, &whi);
            if (final_w)
                for (int x = 0; x < V; ++x)
                    final_w[(size_t)b * V + x] = w[x] / S;
            if (resid_mass) resid_mass[b] = S;
        }
        if (st == ORC_OK) {
            ot[len++] = y;
            out_len[b] = len;
            if (accept_tie) accept_tie[b] = atie;
            if (sample_tie) sample_tie[b] = stie;
            if (sample_lo) sample_lo[b] = T > 0.0 ? wlo : y;
            if (sample_hi) sample_hi[b] = T > 0.0 ? whi : y;
        } else {
            for (int j = 0; j < M; ++j) {
                ot[j] = -1;
                on[j] = -1;
            }
            nerr += 1;
        }
        if (status) status[b] = st != ORC_OK ? st : flags;
        free(zt); free(zd); free(r); free(q); free(w);
    }
    return nerr;
}
