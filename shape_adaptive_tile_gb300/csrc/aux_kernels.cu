// Small kernels around the GEMM: C = beta * C for K == 0 or alpha == 0, the
// registry lookup, and the bounded-wait self-test.
#include <cstdint>

#include "ptx.cuh"
#include "registry.h"

namespace sat {

__global__ void sat_scale_kernel(float* __restrict__ C, long long n, float beta)
{
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        C[i] = beta == 0.0f ? 0.0f : beta * C[i];
}

cudaError_t launch_scale(float* C, long long n, float beta, cudaStream_t stream)
{
    if (n <= 0)
        return cudaSuccess;
    long long blocks = (n + 255) / 256;
    if (blocks > 4096)
        blocks = 4096;
    sat_scale_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(C, n, beta);
    return cudaGetLastError();
}

// Split-K reduction: C[i] = alpha * (W_0[i] + W_1[i] + ... + W_{S-1}[i]) + beta * C[i],
// summed in the fixed order s = 0, 1, ..., S-1 so that the result is the same on
// every run. W_s is slice s of the workspace (`slice` floats apart, same row
// stride N as C). beta == 0 never reads C. Memory-bound: S + 1 (+1) floats
// of traffic per output element.
__global__ void sat_splitk_reduce_kernel(const float* __restrict__ ws, int S, long long slice, float* C, long long n,
                                         float alpha, float beta)
{
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long n4 = (reinterpret_cast<uintptr_t>(C) % 16 == 0 && slice % 4 == 0) ? n / 4 : 0;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
        float4 a = reinterpret_cast<const float4*>(ws)[i];
        for (int s = 1; s < S; ++s) {
            const float4 b = reinterpret_cast<const float4*>(ws + s * slice)[i];
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
        }
        float4 o = make_float4(alpha * a.x, alpha * a.y, alpha * a.z, alpha * a.w);
        if (beta != 0.0f) {
            const float4 c = reinterpret_cast<const float4*>(C)[i];
            o.x = fmaf(beta, c.x, o.x);
            o.y = fmaf(beta, c.y, o.y);
            o.z = fmaf(beta, c.z, o.z);
            o.w = fmaf(beta, c.w, o.w);
        }
        reinterpret_cast<float4*>(C)[i] = o;
    }
    for (long long i = 4 * n4 + static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        float a = ws[i];
        for (int s = 1; s < S; ++s)
            a += ws[s * slice + i];
        float o = alpha * a;
        if (beta != 0.0f)
            o = fmaf(beta, C[i], o);
        C[i] = o;
    }
}

cudaError_t launch_splitk_reduce(const float* ws, int S, long long slice, float* C, long long n, float alpha,
                                 float beta, int sm_count, cudaStream_t stream)
{
    if (n <= 0)
        return cudaSuccess;
    long long blocks = (n / 4 + 255) / 256;
    const long long cap = 8LL * (sm_count > 0 ? sm_count : 1);
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    sat_splitk_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(ws, S, slice, C, n, alpha, beta);
    return cudaGetLastError();
}

// One CTA waits on a barrier that nothing arrives at, through the same
// bounded wait the GEMM kernels use; it must give up after timeout_ns and
// record the timeout bit.
__global__ void sat_wait_probe_kernel(uint32_t* err, unsigned long long timeout_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtl w{&abort_flag, err, timeout_ns};
        wait_bar<false>(smem_u32(&bar), 0, w, 1u << 4);
    }
    __syncthreads();
}

cudaError_t launch_wait_probe(uint32_t* err, unsigned long long timeout_ns, cudaStream_t stream)
{
    sat_wait_probe_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
    return cudaGetLastError();
}

const KernelEntry* find_entry(int dt, int bn, int cg, int prod)
{
    const KernelEntry* tab = dt == kDtTF32 ? kEntriesTF32 : dt == kDtBF16 ? kEntriesBF16 : kEntriesFP16;
    const int n = dt == kDtTF32 ? kNumEntriesTF32 : dt == kDtBF16 ? kNumEntriesBF16 : kNumEntriesFP16;
    for (int i = 0; i < n; ++i)
        if (tab[i].bn == bn && tab[i].cg == cg && tab[i].prod == prod)
            return &tab[i];
    return nullptr;
}

}  // namespace sat
