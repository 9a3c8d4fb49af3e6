// Row operators over a rows x width fp32 matrix: softmax, RMSNorm and
// LayerNorm of each row (include/rowops.h).
//
// These are the wide-row reductions of "Scale coverage exposes a remaining
// GEMM gap" (section "Reductions: wide rows and large working sets"),
// 37 x 8191 to 16384 x 4096. They read each element once and write it once,
// so HBM bandwidth bounds them: 8 bytes per element. One CTA of 128 to 512
// threads takes a row; each thread keeps its PER elements of the row in
// registers between the reductions and the write, so the row is read from
// memory once. Loads are 16 bytes wide where the row start, the row strides
// and the width allow it, 4 bytes otherwise; consecutive threads read
// consecutive addresses either way. Reductions go warp by warp with
// shuffles, then across the CTA's warps through shared memory, in a fixed
// order: the result is the same on every run.
#include "rowops.h"

#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "registry.h"

namespace {


enum Op { kSoftmax = 0, kRMSNorm = 1, kLayerNorm = 2 };

// exp(d) is computed as 2^(d log2 e): exp2f is cheaper than expf, and the
// rounding of d log2 e adds a relative error of about |d| 2^-24 ln 2, below
// 1e-6 for the |d| < 16 of rows of order one. d = 0 still gives exactly 1.
constexpr float kLog2e = 1.4426950408889634f;

// Sum (or maximum) over the block, the same value returned to every thread.
// Consecutive reductions alternate between two scratch rows, so one barrier
// each suffices: a row is rewritten only two reductions later, after a
// barrier that every thread passed after reading it.
template <bool kMax, int NW>
__device__ __forceinline__ float block_reduce(float v, float (*scratch)[NW], int& turn)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float u = __shfl_xor_sync(0xffffffffu, v, o);
        v = kMax ? fmaxf(v, u) : v + u;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* row = scratch[turn];
    turn ^= 1;
    if (lane == 0)
        row[warp] = v;
    __syncthreads();
    float t = lane < NW ? row[lane] : (kMax ? -INFINITY : 0.0f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float u = __shfl_xor_sync(0xffffffffu, t, o);
        t = kMax ? fmaxf(t, u) : t + u;
    }
    return t;
}

// CTAs of NT threads holding PER values each that the launch bounds ask to
// fit on one SM at once: rows of 32 values per thread in 16-byte vectors
// otherwise leave the compiler free to take more registers than two
// 512-thread (three 256-thread) CTAs can share, and an SM then holds one row
// where it could hold two. (The 4-byte variants would spill under that bound;
// 0 leaves the other variants unconstrained.)
template <int NT, int PER, int VEC>
constexpr int kRowMinBlocks = PER == 32 && VEC == 4 ? (NT == 512 ? 2 : NT == 256 ? 3 : 0) : 0;

// NT threads (one CTA) take a row; element e of a thread's share is column
// e / VEC * NT * VEC + threadIdx.x * VEC + e % VEC. VEC = 4 loads 16 bytes
// at a time.
template <int OP, int NT, int PER, int VEC>
__global__ void __launch_bounds__(NT, (kRowMinBlocks<NT, PER, VEC>))
    sat_rowop_kernel(const float* X, int64_t ldx, const float* __restrict__ gamma,
                     const float* __restrict__ beta, float* Y, int64_t ldy, int64_t rows, int width,
                     float eps)
{
    constexpr int NW = NT / 32;  // warps per row
    __shared__ float scratch[2][NW];
    int turn = 0;
    constexpr int NV = PER / VEC;  // vectors per thread
    auto load_row = [&](float(&v)[PER], int64_t r) {
        const float* x = X + r * ldx;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = (i * NT + threadIdx.x) * VEC;
            if constexpr (VEC == 4) {
                float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
                if (c < width)
                    q = *reinterpret_cast<const float4*>(x + c);
                v[4 * i] = q.x;
                v[4 * i + 1] = q.y;
                v[4 * i + 2] = q.z;
                v[4 * i + 3] = q.w;
            } else {
                v[i] = c < width ? x[c] : 0.0f;
            }
        }
    };
    // Rows of 4-byte elements (up to 16 per thread): gamma and beta are read
    // into registers right after the row, so their latency overlaps the
    // row's instead of following the reductions one column at a time.
    constexpr bool kEarly = VEC == 1 && PER <= 16 && OP != kSoftmax;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        float v[PER];
        load_row(v, r);
        float ge[kEarly ? PER : 1], be[kEarly && OP == kLayerNorm ? PER : 1];
        if constexpr (kEarly) {
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int c = i * NT + threadIdx.x;
                ge[i] = gamma && c < width ? gamma[c] : 1.0f;
                if constexpr (OP == kLayerNorm)
                    be[i] = beta && c < width ? beta[c] : 0.0f;
            }
        }
        auto valid = [&](int i) { return (i / VEC * NT + threadIdx.x) * VEC + i % VEC < width; };
        float scale = 0.0f, shift = 0.0f;
        if constexpr (OP == kSoftmax) {
            float m = -INFINITY;
#pragma unroll
            for (int i = 0; i < PER; ++i)
                if (valid(i))
                    m = fmaxf(m, v[i]);
            m = block_reduce<true>(m, scratch, turn);
            float s = 0.0f;
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                v[i] = valid(i) ? exp2f((v[i] - m) * kLog2e) : 0.0f;
                s += v[i];
            }
            s = block_reduce<false>(s, scratch, turn);
            scale = 1.0f / s;
        } else if constexpr (OP == kRMSNorm) {
            float s = 0.0f;
#pragma unroll
            for (int i = 0; i < PER; ++i)
                s = fmaf(v[i], v[i], s);  // padding entries are zero
            s = block_reduce<false>(s, scratch, turn);
            scale = 1.0f / sqrtf(s / static_cast<float>(width) + eps);
        } else {
            float s = 0.0f;
#pragma unroll
            for (int i = 0; i < PER; ++i)
                s += v[i];
            shift = block_reduce<false>(s, scratch, turn) / static_cast<float>(width);
            float q = 0.0f;
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const float d = valid(i) ? v[i] - shift : 0.0f;
                q = fmaf(d, d, q);
            }
            q = block_reduce<false>(q, scratch, turn);
            scale = 1.0f / sqrtf(q / static_cast<float>(width) + eps);
        }
        float* y = Y + r * ldy;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = (i * NT + threadIdx.x) * VEC;
            if (c >= width)
                continue;
            // gamma and beta for these VEC columns, 16 bytes at a time when VEC is 4
            float gv[VEC], bv[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                gv[e] = 1.0f;
                bv[e] = 0.0f;
            }
            if constexpr (kEarly) {
                gv[0] = ge[i];
                if constexpr (OP == kLayerNorm)
                    bv[0] = be[i];
            } else if constexpr (OP != kSoftmax) {
                if (gamma) {
                    if constexpr (VEC == 4) {
                        const float4 q = *reinterpret_cast<const float4*>(gamma + c);
                        gv[0] = q.x, gv[1] = q.y, gv[2] = q.z, gv[3] = q.w;
                    } else {
                        gv[0] = gamma[c];
                    }
                }
                if (OP == kLayerNorm && beta) {
                    if constexpr (VEC == 4) {
                        const float4 q = *reinterpret_cast<const float4*>(beta + c);
                        bv[0] = q.x, bv[1] = q.y, bv[2] = q.z, bv[3] = q.w;
                    } else {
                        bv[0] = beta[c];
                    }
                }
            }
            float o[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float t = v[VEC * i + e];
                if constexpr (OP == kSoftmax)
                    o[e] = t * scale;
                else if constexpr (OP == kRMSNorm)
                    o[e] = t * scale * gv[e];
                else
                    o[e] = fmaf((t - shift) * scale, gv[e], bv[e]);
            }
            if constexpr (VEC == 4)
                *reinterpret_cast<float4*>(y + c) = make_float4(o[0], o[1], o[2], o[3]);
            else
                y[c] = o[0];
        }
    }
}

template <int OP, int NT, int PER, int VEC>
cudaError_t launch_one(const float* X, int64_t ldx, const float* gamma, const float* beta, float* Y, int64_t ldy,
                       int64_t rows, int width, float eps, cudaStream_t stream)
{
    const int64_t grid = rows < 65535 ? rows : 65535;
    sat_rowop_kernel<OP, NT, PER, VEC><<<static_cast<unsigned>(grid), NT, 0, stream>>>(X, ldx, gamma, beta, Y, ldy,
                                                                                       rows, width, eps);
    return cudaGetLastError();
}

template <int OP, int VEC>
cudaError_t launch_vec(const float* X, int64_t ldx, const float* g, const float* b, float* Y, int64_t ldy,
                       int64_t rows, int width, float eps, cudaStream_t s)
{
    // Rows of 16-byte vectors up to 8192 columns: fewer threads per row,
    // each holding more of it. That spreads the per-row work (the
    // reductions, the scale, the index arithmetic) over more elements and
    // keeps more loads in flight per thread; the thread counts are the
    // fastest measured per operator on GB300 (rows x 256 to x 8192).
    if constexpr (VEC == 4) {
        if (width <= 512)
            return launch_one<OP, 128, 4, VEC>(X, ldx, g, b, Y, ldy, rows, width, eps, s);
        if (width <= 1024)
            return launch_one<OP, 128, 8, VEC>(X, ldx, g, b, Y, ldy, rows, width, eps, s);
        if (width <= 2048)
            return launch_one<OP, 128, 16, VEC>(X, ldx, g, b, Y, ldy, rows, width, eps, s);
        if (width <= 4096) {
            if constexpr (OP == kLayerNorm)
                return launch_one<OP, 128, 32, VEC>(X, ldx, g, b, Y, ldy, rows, width, eps, s);
            else
                return launch_one<OP, 256, 16, VEC>(X, ldx, g, b, Y, ldy, rows, width, eps, s);
        }
        if constexpr (OP != kRMSNorm) {
            if (width > 4096 && width <= 8192)
                return launch_one<OP, 256, 32, VEC>(X, ldx, g, b, Y, ldy, rows, width, eps, s);
        }
    }
    // Otherwise 512 threads, with the smallest register share that holds the row.
    if (width <= 512 * 4)
        return launch_one<OP, 512, 4, VEC>(X, ldx, g, b, Y, ldy, rows, width, eps, s);
    if (width <= 512 * 8)
        return launch_one<OP, 512, 8, VEC>(X, ldx, g, b, Y, ldy, rows, width, eps, s);
    if (width <= 512 * 16)
        return launch_one<OP, 512, 16, VEC>(X, ldx, g, b, Y, ldy, rows, width, eps, s);
    if (width <= 512 * 32)
        return launch_one<OP, 512, 32, VEC>(X, ldx, g, b, Y, ldy, rows, width, eps, s);
    return launch_one<OP, 512, 64, VEC>(X, ldx, g, b, Y, ldy, rows, width, eps, s);
}

template <int OP>
int run(const float* X, int64_t ldx, const float* gamma, const float* beta, float* Y, int64_t ldy, int64_t rows,
        int64_t width, float eps, void* stream)
{
    sat::set_last_error("");
    if (rows < 0 || width < 0)
        return sat::fail_with(GEMM_ERR_ARG, "negative size");
    if (rows == 0 || width == 0)
        return GEMM_OK;
    if (width > kRowopMaxWidth)
        return sat::fail_with(GEMM_ERR_ARG, "width %lld is above the %d these kernels hold in registers",
                              (long long)width,
                    kRowopMaxWidth);
    if (!X || !Y)
        return sat::fail_with(GEMM_ERR_ARG, "X or Y is NULL");
    if (ldx < width || ldy < width)
        return sat::fail_with(GEMM_ERR_ARG, "row stride below the width");
    if (reinterpret_cast<uintptr_t>(X) % 4 || reinterpret_cast<uintptr_t>(Y) % 4 ||
        (gamma && reinterpret_cast<uintptr_t>(gamma) % 4) || (beta && reinterpret_cast<uintptr_t>(beta) % 4))
        return sat::fail_with(GEMM_ERR_ALIGN, "operands must be 4-byte aligned");
    auto al16 = [](const void* p) { return p == nullptr || reinterpret_cast<uintptr_t>(p) % 16 == 0; };
    const bool vec = width % 4 == 0 && ldx % 4 == 0 && ldy % 4 == 0 && al16(X) && al16(Y) && al16(gamma) &&
                     al16(beta);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int w = static_cast<int>(width);
    const cudaError_t e = vec ? launch_vec<OP, 4>(X, ldx, gamma, beta, Y, ldy, rows, w, eps, s)
                              : launch_vec<OP, 1>(X, ldx, gamma, beta, Y, ldy, rows, w, eps, s);
    return e == cudaSuccess ? GEMM_OK
                            : sat::fail_with(GEMM_ERR_LAUNCH, "launching the row kernel: %s", cudaGetErrorString(e));
}

}  // namespace

extern "C" {

int rowop_softmax(const float* X, int64_t ldx, float* Y, int64_t ldy, int64_t rows, int64_t width, void* stream)
{
    return run<kSoftmax>(X, ldx, nullptr, nullptr, Y, ldy, rows, width, 0.0f, stream);
}

int rowop_rmsnorm(const float* X, int64_t ldx, const float* gamma, float* Y, int64_t ldy, int64_t rows, int64_t width,
                  float eps, void* stream)
{
    return run<kRMSNorm>(X, ldx, gamma, nullptr, Y, ldy, rows, width, eps, stream);
}

int rowop_layernorm(const float* X, int64_t ldx, const float* gamma, const float* beta, float* Y, int64_t ldy,
                    int64_t rows, int64_t width, float eps, void* stream)
{
    return run<kLayerNorm>(X, ldx, gamma, beta, Y, ldy, rows, width, eps, stream);
}

}  // extern "C"
