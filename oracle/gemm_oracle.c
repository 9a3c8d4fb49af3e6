/*
 * FP64 CPU oracle for the dense GEMM  C = alpha * A * B + beta * C0.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may include, link
 * or call this file: only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark use it. It shares no source with the CUDA library.
 *
 * What it computes, and where the definition comes from:
 *   - "Post-mortem: a GPU stack without nvcc, cuBLAS, or LLVM", section 5
 *     ("Compiling clean is not being correct") and section 11 item 4: every
 *     GPU kernel is gated on numerics against an f64 CPU reference.
 *   - "Scale coverage exposes a remaining GEMM gap", section "Measurement
 *     contract and evidence": GEMM is C = A*B over compact row-major inputs,
 *     no transpose, checked on the complete output; its dyadic input family
 *     gives exact results.
 *   - The alpha/beta form is the BLAS definition of GEMM: C = alpha*A*B +
 *     beta*C0, and beta == 0 means C0 is not read (so a NaN there is
 *     ignored).
 *
 * Element (i, j) is the plain definition written out:
 *     acc    = sum_{k = 0, 1, ..., K-1} A[i][k] * B[k][j]   (ascending k,
 *              each product and each sum rounded to double)
 *     out64  = alpha * acc + beta * C0[i][j]                 (in double)
 *     out32  = (float) out64                                 (one rounding,
 *              to nearest even)
 * A and B enter as the exact values of the stored bits (fp32, bf16 or fp16
 * are all exact in double). The full-matrix routine walks i-k-j with a
 * double row accumulator; for fixed (i, j) this is the same ascending-k
 * sequence of operations as the i-j-k textbook loop, so both give the same
 * bits. Build with -ffp-contract=off so no product is fused into a sum.
 *
 * Operand element types (own codes, not shared with the library):
 *   0 = fp32 (the GPU computes it in TF32; the oracle uses the full fp32
 *       value), 1 = bf16 (bit patterns, uint16), 2 = fp16 (uint16).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1, OR_F16 = 2 };

/* Exact value of a stored element, decoded from the IEEE-754 field layout
 * of each format (binary16: 1/5/10 bits, bias 15; bfloat16: 1/8/7 bits,
 * bias 127), not by reinterpreting memory. */
static double decode_bits(int dtype, uint32_t bits)
{
    if (dtype == OR_F32) {
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    int ebits = dtype == OR_F16 ? 5 : 8;
    int fbits = dtype == OR_F16 ? 10 : 7;
    int bias = (1 << (ebits - 1)) - 1;
    uint32_t sign = (bits >> (ebits + fbits)) & 1u;
    uint32_t e = (bits >> fbits) & ((1u << ebits) - 1u);
    uint32_t f = bits & ((1u << fbits) - 1u);
    double v;
    if (e == 0)                       /* zero or subnormal: f * 2^(1-bias-fbits) */
        v = ldexp((double)f, 1 - bias - fbits);
    else if (e == (1u << ebits) - 1u) /* infinity or NaN */
        v = f ? NAN : INFINITY;
    else                              /* normal: (2^fbits + f) * 2^(e-bias-fbits) */
        v = ldexp((double)((1u << fbits) + f), (int)e - bias - fbits);
    return sign ? -v : v;
}

static double load(int dtype, const void* p, int64_t idx)
{
    if (dtype == OR_F32) {
        uint32_t b;
        memcpy(&b, (const char*)p + 4 * idx, 4);
        return decode_bits(OR_F32, b);
    }
    return decode_bits(dtype, ((const uint16_t*)p)[idx]);
}

double oracle_decode(int dtype, uint32_t bits) { return decode_bits(dtype, bits); }

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int bad_args(int64_t M, int64_t N, int64_t K, int dtype)
{
    return M < 0 || N < 0 || K < 0 || dtype < OR_F32 || dtype > OR_F16;
}

/* Rows [row_begin, row_end) of the full result; out64/out32 are
 * (row_end - row_begin) x N row-major (either may be NULL). Returns 0, or
 * -1 on bad arguments, -2 on allocation failure. */
int oracle_gemm_rows(int64_t M, int64_t N, int64_t K, int dtype,
                     const void* A, const void* B, const float* C0,
                     double alpha, double beta,
                     int64_t row_begin, int64_t row_end,
                     double* out64, float* out32)
{
    if (bad_args(M, N, K, dtype) || row_begin < 0 || row_end > M || row_begin > row_end)
        return -1;
    if (row_begin == row_end || N == 0)
        return 0;
    double* Bd = (double*)malloc(sizeof(double) * (size_t)(K * N > 0 ? K * N : 1));
    if (!Bd)
        return -2;
    for (int64_t t = 0; t < K * N; ++t)
        Bd[t] = load(dtype, B, t);
    int fail = 0;
#pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)N);
        double* arow = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        if (!acc || !arow) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = row_begin; i < row_end; ++i) {
                for (int64_t k = 0; k < K; ++k)
                    arow[k] = load(dtype, A, i * K + k);
                for (int64_t j = 0; j < N; ++j)
                    acc[j] = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    const double a = arow[k];
                    const double* brow = Bd + k * N;
                    for (int64_t j = 0; j < N; ++j)
                        acc[j] = acc[j] + a * brow[j];
                }
                for (int64_t j = 0; j < N; ++j) {
                    double v = alpha * acc[j];
                    if (beta != 0.0)
                        v = v + beta * (double)C0[i * N + j];
                    const int64_t o = (i - row_begin) * N + j;
                    if (out64)
                        out64[o] = v;
                    if (out32)
                        out32[o] = (float)v;
                }
            }
        }
        free(acc);
        free(arow);
    }
    free(Bd);
    return fail ? -2 : 0;
}

int oracle_gemm(int64_t M, int64_t N, int64_t K, int dtype,
                const void* A, const void* B, const float* C0,
                double alpha, double beta, double* out64, float* out32)
{
    return oracle_gemm_rows(M, N, K, dtype, A, B, C0, alpha, beta, 0, M, out64, out32);
}

/* Selected entries (rows[e], cols[e]), e = 0..n-1, each by the same
 * ascending-k definition as above; for checking very large problems. */
int oracle_gemm_entries(int64_t M, int64_t N, int64_t K, int dtype,
                        const void* A, const void* B, const float* C0,
                        double alpha, double beta,
                        int64_t n, const int64_t* rows, const int64_t* cols,
                        double* out64, float* out32)
{
    if (bad_args(M, N, K, dtype) || n < 0)
        return -1;
    for (int64_t e = 0; e < n; ++e)
        if (rows[e] < 0 || rows[e] >= M || cols[e] < 0 || cols[e] >= N)
            return -1;
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < n; ++e) {
        const int64_t i = rows[e], j = cols[e];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc = acc + load(dtype, A, i * K + k) * load(dtype, B, k * N + j);
        double v = alpha * acc;
        if (beta != 0.0)
            v = v + beta * (double)C0[i * N + j];
        if (out64)
            out64[e] = v;
        if (out32)
            out32[e] = (float)v;
    }
    return 0;
}
