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
