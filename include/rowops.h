/*
 * Row operators over a rows x width fp32 matrix, one row at a time: softmax,
 * RMSNorm and LayerNorm. The C ABI of the library's second workload.
 *
 * "Scale coverage exposes a remaining GEMM gap" (section "Reductions: wide
 * rows and large working sets") times these three operators on rows x width
 * from 37 x 8191 to 16384 x 4096, in fp32. The page names them without
 * formulas; these are the textbook ones:
 *   softmax:   y_j = exp(x_j - max_k x_k) / sum_k exp(x_k - max_k x_k)
 *   RMSNorm:   y_j = x_j / sqrt(mean_k x_k^2 + eps) * gamma_j
 *   LayerNorm: y_j = (x_j - mu) / sqrt(var + eps) * gamma_j + beta_j,
 *              mu = mean_k x_k, var = mean_k (x_k - mu)^2 (biased)
 * gamma and beta may be NULL (taken as 1 and 0).
 *
 * X and Y are device pointers to rows x width floats with row strides ldx
 * and ldy (>= width); Y may be X (in place, same stride). Reductions are in
 * fp32 in a fixed order, so results are identical from run to run. The
 * calls enqueue one kernel on `stream` and return without synchronising;
 * they return 0 or a negative gemm_status_t (message in gemm_last_error):
 * GEMM_ERR_ARG for negative sizes, NULL X/Y, strides below the width or a
 * width above ROWOP_MAX_WIDTH; GEMM_ERR_ALIGN for pointers not 4-byte
 * aligned. rows == 0 or width == 0 does nothing.
 */
#ifndef SAT_ROWOPS_H
#define SAT_ROWOPS_H

#include <stdint.h>

#include "gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Widest row the kernels hold (512 threads x 64 values in registers). */
#define ROWOP_MAX_WIDTH 32768

int rowop_softmax(const float* X, int64_t ldx, float* Y, int64_t ldy, int64_t rows, int64_t width, void* stream);

int rowop_rmsnorm(const float* X, int64_t ldx, const float* gamma, float* Y, int64_t ldy, int64_t rows, int64_t width,
                  float eps, void* stream);

int rowop_layernorm(const float* X, int64_t ldx, const float* gamma, const float* beta, float* Y, int64_t ldy,
                    int64_t rows, int64_t width, float eps, void* stream);

#ifdef __cplusplus
}
#endif

#ifdef __cplusplus
constexpr int kRowopMaxWidth = ROWOP_MAX_WIDTH;
#endif

#endif
