/*
 * FP64 CPU oracle for the row operators: softmax, RMSNorm and LayerNorm over
 * each row of a rows x width fp32 matrix (row stride ld floats).
 *
 * TEST INFRASTRUCTURE ONLY (see oracle/__init__.py). Plain loops in double,
 * every sum taken in ascending column order; no blocking or reordering.
 *
 * The operators are those whose wide-row cases "Scale coverage exposes a
 * remaining GEMM gap" times (section "Reductions: wide rows and large
 * working sets": softmax, RMSNorm and LayerNorm, rows x width from 37 x 8191
 * to 16384 x 4096). The page names them without formulas; the textbook
 * definitions are written out here:
 *   softmax:   y_j = exp(x_j - max_k x_k) / sum_k exp(x_k - max_k x_k)
 *   RMSNorm:   y_j = x_j / sqrt(mean_k x_k^2 + eps) * gamma_j
 *   LayerNorm: y_j = (x_j - mu) / sqrt(var + eps) * gamma_j + beta_j,
 *              mu = mean_k x_k, var = mean_k (x_k - mu)^2 (biased)
 * gamma and beta may be NULL (taken as 1 and 0).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

void oracle_softmax_rows(const float* x, int64_t ld, int64_t rows, int64_t width, double* y)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * ld;
        double* yr = y + r * width;
        double m = -INFINITY;
        for (int64_t j = 0; j < width; ++j)
            if ((double)xr[j] > m)
                m = (double)xr[j];
        double s = 0.0;
        for (int64_t j = 0; j < width; ++j) {
            yr[j] = exp((double)xr[j] - m);
            s += yr[j];
        }
        for (int64_t j = 0; j < width; ++j)
            yr[j] /= s;
    }
}

void oracle_rmsnorm_rows(const float* x, int64_t ld, const float* gamma, int64_t rows, int64_t width, double eps,
                         double* y)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * ld;
        double ss = 0.0;
        for (int64_t j = 0; j < width; ++j)
            ss += (double)xr[j] * (double)xr[j];
        const double inv = 1.0 / sqrt(ss / (double)width + eps);
        for (int64_t j = 0; j < width; ++j)
            y[r * width + j] = (double)xr[j] * inv * (gamma ? (double)gamma[j] : 1.0);
    }
}

void oracle_layernorm_rows(const float* x, int64_t ld, const float* gamma, const float* beta, int64_t rows,
                           int64_t width, double eps, double* y)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * ld;
        double s = 0.0;
        for (int64_t j = 0; j < width; ++j)
            s += (double)xr[j];
        const double mu = s / (double)width;
        double v = 0.0;
        for (int64_t j = 0; j < width; ++j) {
            const double d = (double)xr[j] - mu;
            v += d * d;
        }
        const double inv = 1.0 / sqrt(v / (double)width + eps);
        for (int64_t j = 0; j < width; ++j)
            y[r * width + j] =
                ((double)xr[j] - mu) * inv * (gamma ? (double)gamma[j] : 1.0) + (beta ? (double)beta[j] : 0.0);
    }
}
