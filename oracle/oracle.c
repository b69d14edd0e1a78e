/*
 * Fused LM-head loss: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  It shares no code,
 * header, table or helper with the CUDA library, and neither side includes the
 * other.  Every quantity is computed from its plain definition in double
 * precision, one row at a time, with no blocking, fusion or reordering.
 *
 * Sources (page title, then the section the formula comes from):
 *  [TT]  torchtitan PR 5661 "fix softmax collapse with improved CE perf":
 *        commit message, "Numerics (TP > 1 only)": NLL = softplus(lse_{j!=t} z_j - z_t),
 *        the target term dropped before the sum, target gradient p_t - 1 below
 *        p_t = 1/4 else -p_non_target; review "Example": the margin-20 row.
 *  [XT]  xtuner PR 1963 "[FSDP][Loss] Switch gradient reduction to SUM":
 *        description (each rank's loss is its local component; SUM of the
 *        components is the global token-mean) and the z-loss diff
 *        (loss * z_loss_alpha / batch_size).
 *  [FL]  Fast-LLM PR 552 "Fuse GSPO into the monolithic compiled loss (#507)":
 *        "Why it needed special handling" (segment index_add over num_segments,
 *        then clipping) and the list of combinable losses (CE, z-loss,
 *        distillation, GRPO).
 *
 * The pages leave the distillation and GSPO formulas open; the readings used
 * here are the plainest ones consistent with them:
 *  - distillation = forward KL(teacher || student) at temperature tau,
 *    KL = sum_j q_j (log q_j - log p^tau_j), q = softmax(u / tau),
 *    p^tau = softmax(z / tau); gradient (p^tau - q) / tau, no tau^2 factor;
 *  - GSPO per segment i: n_i active tokens, D_i = sum (logp_t - old_logp),
 *    s_i = exp(D_i / n_i), L_i = -min(s_i A_i, clamp(s_i, 1-eps_lo, 1+eps_hi) A_i);
 *    its gradient flows through s_i only when s_i A_i <= clamp(s_i) A_i.
 *    (The segment seam itself lives in oracle.py; this file supplies the rows.)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_BF16 = 0, ORC_FP32 = 1 };

/* One logit, widened exactly to double.  bf16 is the top half of an fp32. */
static double orc_elem(int dtype, const void* base, int64_t idx)
{
    if (dtype == ORC_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float*)base)[idx];
}

/* log(sum_{j != skip} exp(x_j)), shifted by its own maximum over the same set.
 * An empty set, or one holding only -inf, gives -inf. */
static double orc_logsumexp_skip(const double* x, int64_t n, int64_t skip)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (j != skip && x[j] > m) m = x[j];
    if (m == -INFINITY) {
        for (int64_t j = 0; j < n; ++j)   /* NaN anywhere in the set stays NaN */
            if (j != skip && isnan(x[j])) return NAN;
        return -INFINITY;
    }
    double s = 0.0;
    for (int64_t j = 0; j < n; ++j)
        if (j != skip) s += exp(x[j] - m);
    return m + log(s);
}

/* softplus(x) = log(1 + e^x), in the form that loses nothing at either end. */
static double orc_softplus(double x)
{
    if (x > 0.0) return x + log1p(exp(-x));
    return log1p(exp(x));
}

/* log(e^a + e^b). */
static double orc_logaddexp(double a, double b)
{
    if (a == -INFINITY && b == -INFINITY) return -INFINITY;
    double hi = a > b ? a : b;
    double lo = a > b ? b : a;
    if (isnan(a) || isnan(b)) return NAN;
    return hi + log1p(exp(lo - hi));
}

typedef struct {
    double nll;     /* softplus(lse_nt - z_t)                                  */
    double lse;     /* log sum_j exp(z_j)                                      */
    double lse_nt;  /* log sum_{j != t} exp(z_j)                               */
    double kl;      /* KL(teacher || student) at temperature tau, 0 if none    */
} orc_row_stats;

/* Per-row scalars for one active row: z[0..V) logits, t the target column,
 * u[0..V) teacher logits or NULL.  [TT] Numerics: the non-target logsumexp is
 * formed with the target excluded from the sum (not subtracted from it), and
 * the NLL is its softplus against z_t. */
static orc_row_stats orc_row_forward(const double* z, const double* u, int64_t V,
                                     int64_t t, double tau, double* work)
{
    orc_row_stats r;
    r.lse_nt = orc_logsumexp_skip(z, V, t);
    r.nll = orc_softplus(r.lse_nt - z[t]);
    r.lse = orc_logaddexp(z[t], r.lse_nt);
    r.kl = 0.0;
    if (u) {
        /* q = softmax(u/tau), p^tau = softmax(z/tau) */
        double* a = work;        /* u / tau */
        double* b = work + V;    /* z / tau */
        for (int64_t j = 0; j < V; ++j) { a[j] = u[j] / tau; b[j] = z[j] / tau; }
        double lse_a = orc_logsumexp_skip(a, V, -1);
        double lse_b = orc_logsumexp_skip(b, V, -1);
        double kl = 0.0;
        for (int64_t j = 0; j < V; ++j) {
            double log_q = a[j] - lse_a;
            double q = exp(log_q);
            if (q == 0.0) continue;            /* 0 * log 0 = 0 */
            kl += q * (log_q - (b[j] - lse_b));
        }
        r.kl = kl;
    }
    return r;
}

static void orc_load_row(int dtype, const void* base, int64_t r, int64_t V, int64_t ld, double* out)
{
    for (int64_t j = 0; j < V; ++j) out[j] = orc_elem(dtype, base, r * ld + j);
}

static int orc_threads(int nthreads)
{
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/*
 * Forward scalars for n consecutive rows of logits [n, ld] (first V columns
 * used).  Inactive rows (active[r] == 0) get 0 everywhere.  Targets of active
 * rows must lie in [0, V).  Rows are independent; the parallel loop over rows
 * changes no arithmetic.  Returns 0, or -1 when scratch cannot be allocated.
 */
int orc_forward(int dtype, int64_t n, int64_t V, int64_t ld,
                const void* logits, const void* teacher, double temperature,
                const int64_t* targets, const uint8_t* active,
                double* nll, double* lse, double* lse_nt, double* kl, int nthreads)
{
    int failed = 0;
#pragma omp parallel num_threads(orc_threads(nthreads))
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
        double* u = teacher ? (double*)malloc(sizeof(double) * (size_t)V) : NULL;
        double* work = teacher ? (double*)malloc(sizeof(double) * 2 * (size_t)V) : NULL;
        int ok = z && (!teacher || (u && work));
        if (!ok) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < n; ++r) {
            if (!ok) continue;
            if (!active[r]) {
                nll[r] = lse[r] = lse_nt[r] = kl[r] = 0.0;
                continue;
            }
            orc_load_row(dtype, logits, r, V, ld, z);
            if (teacher) orc_load_row(dtype, teacher, r, V, ld, u);
            orc_row_stats s = orc_row_forward(z, teacher ? u : NULL, V, targets[r], temperature, work);
            nll[r] = s.nll;
            lse[r] = s.lse;
            lse_nt[r] = s.lse_nt;
            kl[r] = s.kl;
        }
        free(z);
        free(u);
        free(work);
    }
    return failed ? -1 : 0;
}

/*
 * Gradient of the total loss with respect to the logits of n consecutive rows,
 * written to grad [n, V] in double.  For an active row r with target t:
 *
 *   g_j = s_tok * ( w_ce * (p_j - [j==t])          cross-entropy
 *                 + 2 * alpha * lse * p_j           z-loss alpha * lse^2   [XT]
 *                 + w_kl * (p^tau_j - q_j) / tau )  distillation           [FL]
 *       + c[r] * (p_j - [j==t])                     GSPO, c[r] from the seam
 *
 * with p = softmax(z).  At the target column, p_t - 1 equals -p_non_target =
 * -exp(lse_nt - lse) in exact arithmetic; that form is used because p_t - 1
 * cancels to 0 in double once the target dominates ([TT] Numerics).
 * Inactive rows get an all-zero gradient.  c may be NULL (no GSPO term).
 * gscale (optional, [n, V]) receives the sum of the magnitudes of the terms
 * above, the scale against which a rounding error in any one term is judged.
 */
int orc_grad(int dtype, int64_t n, int64_t V, int64_t ld,
             const void* logits, const void* teacher, double temperature,
             const int64_t* targets, const uint8_t* active,
             double s_tok, double w_ce, double alpha, double w_kl, const double* c,
             double* grad, double* gscale, int nthreads)
{
    int failed = 0;
#pragma omp parallel num_threads(orc_threads(nthreads))
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
        double* u = teacher ? (double*)malloc(sizeof(double) * (size_t)V) : NULL;
        double* work = teacher ? (double*)malloc(sizeof(double) * 2 * (size_t)V) : NULL;
        int ok = z && (!teacher || (u && work));
        if (!ok) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < n; ++r) {
            double* g = grad + r * V;
            double* gs = gscale ? gscale + r * V : NULL;
            if (!ok) continue;
            if (!active[r]) {
                for (int64_t j = 0; j < V; ++j) g[j] = 0.0;
                if (gs)
                    for (int64_t j = 0; j < V; ++j) gs[j] = 0.0;
                continue;
            }
            int64_t t = targets[r];
            orc_load_row(dtype, logits, r, V, ld, z);
            if (teacher) orc_load_row(dtype, teacher, r, V, ld, u);
            orc_row_stats s = orc_row_forward(z, teacher ? u : NULL, V, t, temperature, work);
            double c_r = c ? c[r] : 0.0;

            double lse_a = 0.0, lse_b = 0.0;
            if (teacher) {
                for (int64_t j = 0; j < V; ++j) { work[j] = u[j] / temperature; work[V + j] = z[j] / temperature; }
                lse_a = orc_logsumexp_skip(work, V, -1);
                lse_b = orc_logsumexp_skip(work + V, V, -1);
            }
            for (int64_t j = 0; j < V; ++j) {
                double p = exp(z[j] - s.lse);
                double p_minus_onehot = (j == t) ? -exp(s.lse_nt - s.lse) : p;
                double term = w_ce * p_minus_onehot + 2.0 * alpha * s.lse * p;
                double mag = fabs(w_ce * p_minus_onehot) + fabs(2.0 * alpha * s.lse * p);
                if (teacher) {
                    double p_tau = exp(work[V + j] - lse_b);
                    double q = exp(work[j] - lse_a);
                    term += w_kl * (p_tau - q) / temperature;
                    mag += fabs(w_kl * p_tau / temperature) + fabs(w_kl * q / temperature);
                }
                g[j] = s_tok * term + c_r * p_minus_onehot;
                if (gs) gs[j] = fabs(s_tok) * mag + fabs(c_r * p_minus_onehot);
            }
        }
        free(z);
        free(u);
        free(work);
    }
    return failed ? -1 : 0;
}

/*
 * Entropy of the softmax of each active row, H = -sum_j p_j log p_j with
 * p = softmax(z), written to ent[r] (0 on inactive rows).  A side output a
 * caller may want next to the loss (torchtitan PR 5661, review "Details":
 * callers reuse the logits, e.g. for entropy).
 */
int orc_entropy(int dtype, int64_t n, int64_t V, int64_t ld, const void* logits,
                const uint8_t* active, double* ent, int nthreads)
{
    int failed = 0;
#pragma omp parallel num_threads(orc_threads(nthreads))
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
        if (!z) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < n; ++r) {
            if (!z) continue;
            if (!active[r]) { ent[r] = 0.0; continue; }
            orc_load_row(dtype, logits, r, V, ld, z);
            /* -log p_j = lse - z_j.  For the largest entry k that difference is
             * log(1 + t), t = sum_{j != k} exp(z_j - z_k), which fp64 would round
             * to 0 as lse - z_k once p_k is within 1e-16 of 1; take it through
             * log1p, and lse - z_j = (z_k - z_j) + log1p(t) for the others. */
            int64_t k = 0;
            for (int64_t j = 1; j < V; ++j)
                if (z[j] > z[k]) k = j;
            double h = 0.0;
            if (z[k] > -INFINITY) {
                double t = 0.0;
                for (int64_t j = 0; j < V; ++j)
                    if (j != k) t += exp(z[j] - z[k]);
                const double l1 = log1p(t);
                for (int64_t j = 0; j < V; ++j) {
                    double nlogp = (j == k) ? l1 : (z[k] - z[j]) + l1;
                    double p = exp(-nlogp);
                    if (p == 0.0) continue;          /* 0 log 0 = 0 */
                    h += p * nlogp;
                }
            }
            ent[r] = h;
        }
        free(z);
    }
    return failed ? -1 : 0;
}
