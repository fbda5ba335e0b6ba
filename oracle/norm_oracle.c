/*
 * norm_oracle.c -- plain fp64 CPU oracle for row-wise RMSNorm and LayerNorm,
 * forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  It shares no code,
 * header, table or helper with the CUDA path, and includes nothing from it.
 *
 * Inputs arrive as double arrays holding values that were already rounded to
 * the storage dtype (bf16, fp16 or fp32); the promotion to double is exact.
 * Every step below is computed in double, row by row, exactly as the
 * definitions read; nothing is blocked, fused or reordered.
 *
 * Sources (web pages):
 *  - "SOTA normalization performance with torch.compile", section
 *    "How Did Torch.compile Catch Quack?": LayerNorm subtracts the row mean,
 *    divides by the standard deviation, then scales by gamma and adds beta;
 *    RMSNorm skips the mean, divides by the root mean square and scales by
 *    gamma.  The backward section of the same page names the outputs: dX,
 *    dW (gamma) and dB (beta), with reductions over dY.
 *  - "Fused RMSNorm", section "What it is": the RMSNorm steps are a square,
 *    a mean, an add (of eps), a reciprocal square root, a multiply (by that
 *    factor) and another multiply (by gamma).
 *
 * Readings where the pages are silent:
 *  - eps is added to the mean square (RMSNorm) or to the variance
 *    (LayerNorm) under the square root.
 *  - The variance is the biased one, (1/N) * sum (x - mean)^2, computed in
 *    two passes (mean first, then the centred squares).
 *  - The backward formulas are the analytic gradients of the forward with
 *    respect to x, gamma and beta (the pages name them, not their form):
 *      xhat_j = (x_j - mean) * rstd       (mean = 0 for RMSNorm)
 *      g_j    = dy_j * gamma_j
 *      RMSNorm:   dx_j = rstd * (g_j - xhat_j * (1/N) sum_k g_k xhat_k)
 *      LayerNorm: dx_j = rstd * (g_j - (1/N) sum_k g_k
 *                                    - xhat_j * (1/N) sum_k g_k xhat_k)
 *      dgamma_j = sum_i dy_ij * xhat_ij,   dbeta_j = sum_i dy_ij.
 *  - The backward recomputes mean and rstd itself, in fp64, from x; it never
 *    reads statistics produced elsewhere.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of host threads the oracle uses (1 when built without OpenMP). */
int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Mean square of one row: (1/N) * sum_j x_j^2.  ("a square, a mean") */
static double row_mean_square(const double *x, int64_t N)
{
    double s = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        double v = x[j];
        s += v * v;
    }
    return s / (double)N;
}

/* Row mean: (1/N) * sum_j x_j. */
static double row_mean(const double *x, int64_t N)
{
    double s = 0.0;
    for (int64_t j = 0; j < N; ++j) s += x[j];
    return s / (double)N;
}

/* Biased variance about a given mean: (1/N) * sum_j (x_j - mean)^2. */
static double row_variance(const double *x, int64_t N, double mean)
{
    double s = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        double d = x[j] - mean;
        s += d * d;
    }
    return s / (double)N;
}

/*
 * RMSNorm forward, per row i:
 *   ms = (1/N) sum_j x_j^2;  rstd = 1 / sqrt(ms + eps);  y_j = (x_j * rstd) * gamma_j.
 * rstd may be NULL.
 */
void oracle_rmsnorm_fwd(const double *x, const double *gamma, int64_t M, int64_t N,
                        double eps, double *y, double *rstd)
{
    int64_t i;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (i = 0; i < M; ++i) {
        const double *xr = x + i * N;
        double ms = row_mean_square(xr, N);
        double r = 1.0 / sqrt(ms + eps);
        double *yr = y + i * N;
        for (int64_t j = 0; j < N; ++j) yr[j] = (xr[j] * r) * gamma[j];
        if (rstd) rstd[i] = r;
    }
}

/*
 * LayerNorm forward, per row i:
 *   mean = (1/N) sum_j x_j;  var = (1/N) sum_j (x_j - mean)^2;
 *   rstd = 1 / sqrt(var + eps);  y_j = ((x_j - mean) * rstd) * gamma_j + beta_j.
 * mean_out and rstd may be NULL.
 */
void oracle_layernorm_fwd(const double *x, const double *gamma, const double *beta,
                          int64_t M, int64_t N, double eps, double *y,
                          double *mean_out, double *rstd)
{
    int64_t i;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (i = 0; i < M; ++i) {
        const double *xr = x + i * N;
        double mu = row_mean(xr, N);
        double var = row_variance(xr, N, mu);
        double r = 1.0 / sqrt(var + eps);
        double *yr = y + i * N;
        for (int64_t j = 0; j < N; ++j)
            yr[j] = ((xr[j] - mu) * r) * gamma[j] + beta[j];
        if (mean_out) mean_out[i] = mu;
        if (rstd) rstd[i] = r;
    }
}

/*
 * Shared body of the two backwards.  is_ln selects LayerNorm (centre by the
 * mean, subtract mean(g)) or RMSNorm (no centring).  dx, dgamma and dbeta may
 * each be NULL; dbeta is only written for LayerNorm.
 */
static int norm_bwd(int is_ln, const double *dy, const double *x, const double *gamma,
                     int64_t M, int64_t N, double eps, double *dx, double *dgamma,
                     double *dbeta)
{
    double *mean = (double *)malloc((size_t)(M > 0 ? M : 1) * sizeof(double));
    double *rstd = (double *)malloc((size_t)(M > 0 ? M : 1) * sizeof(double));
    if (!mean || !rstd) {
        free(mean);
        free(rstd);
        return -1;
    }
    int64_t i;

    /* Pass 1, per row: statistics, then dx. */
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (i = 0; i < M; ++i) {
        const double *xr = x + i * N;
        const double *dyr = dy + i * N;
        double mu, r;
        if (is_ln) {
            mu = row_mean(xr, N);
            r = 1.0 / sqrt(row_variance(xr, N, mu) + eps);
        } else {
            mu = 0.0;
            r = 1.0 / sqrt(row_mean_square(xr, N) + eps);
        }
        mean[i] = mu;
        rstd[i] = r;
        if (!dx) continue;

        double mean_g = 0.0;     /* (1/N) sum_k g_k          */
        double mean_gxhat = 0.0; /* (1/N) sum_k g_k xhat_k   */
        for (int64_t k = 0; k < N; ++k) {
            double xhat = (xr[k] - mu) * r;
            double g = dyr[k] * gamma[k];
            mean_g += g;
            mean_gxhat += g * xhat;
        }
        mean_g /= (double)N;
        mean_gxhat /= (double)N;

        double *dxr = dx + i * N;
        for (int64_t j = 0; j < N; ++j) {
            double xhat = (xr[j] - mu) * r;
            double g = dyr[j] * gamma[j];
            double inner = is_ln ? (g - mean_g - xhat * mean_gxhat) : (g - xhat * mean_gxhat);
            dxr[j] = r * inner;
        }
    }

    /* Pass 2, per column: dgamma_j = sum_i dy_ij xhat_ij and dbeta_j = sum_i dy_ij,
     * each summed over rows in ascending i.  Columns are independent, so they
     * are split across threads in chunks; each column's order is unchanged. */
    if (dgamma || (is_ln && dbeta)) {
        const int64_t CH = 64;
        int64_t nchunks = (N + CH - 1) / CH;
        int64_t c;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
        for (c = 0; c < nchunks; ++c) {
            int64_t j0 = c * CH;
            int64_t j1 = j0 + CH < N ? j0 + CH : N;
            double accg[64], accb[64];
            for (int64_t j = j0; j < j1; ++j) {
                accg[j - j0] = 0.0;
                accb[j - j0] = 0.0;
            }
            for (int64_t ii = 0; ii < M; ++ii) {
                const double *xr = x + ii * N;
                const double *dyr = dy + ii * N;
                for (int64_t j = j0; j < j1; ++j) {
                    double xhat = (xr[j] - mean[ii]) * rstd[ii];
                    accg[j - j0] += dyr[j] * xhat;
                    accb[j - j0] += dyr[j];
                }
            }
            for (int64_t j = j0; j < j1; ++j) {
                if (dgamma) dgamma[j] = accg[j - j0];
                if (is_ln && dbeta) dbeta[j] = accb[j - j0];
            }
        }
    }
    free(mean);
    free(rstd);
    return 0;
}

/* RMSNorm backward: dx [M,N] and dgamma [N] (either may be NULL).
 * Returns 0, or -1 if host memory for the statistics could not be had. */
int oracle_rmsnorm_bwd(const double *dy, const double *x, const double *gamma, int64_t M,
                        int64_t N, double eps, double *dx, double *dgamma)
{
    return norm_bwd(0, dy, x, gamma, M, N, eps, dx, dgamma, NULL);
}

/* LayerNorm backward: dx [M,N], dgamma [N] and dbeta [N] (each may be NULL).
 * Returns 0, or -1 if host memory for the statistics could not be had. */
int oracle_layernorm_bwd(const double *dy, const double *x, const double *gamma, int64_t M,
                          int64_t N, double eps, double *dx, double *dgamma, double *dbeta)
{
    return norm_bwd(1, dy, x, gamma, M, N, eps, dx, dgamma, dbeta);
}
