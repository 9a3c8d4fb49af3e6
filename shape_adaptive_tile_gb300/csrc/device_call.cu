// gemm_selftest_device_call: the device-callable GEMM routine (gemm_cta)
// inside a kernel of its own, as one phase of a persistent kernel.
//
// "Measured data point on fixed-tile vs shape-adaptive GEMM" (section "The
// wall, and why we think it's structural") names the property a host API
// lacks: a GEMM that a persistent megakernel can call inline. This kernel is
// the smallest such megakernel: phase 1 is the GEMM schedule of gemm_cta;
// phase 2, in the same launch, applies max(x, 0) to the tiles of C that this
// CTA has just produced, reading them back from memory. Nothing between the
// phases is a launch boundary: the routine returns with its stores complete
// and ordered for the caller's generic accesses.
#include "gemm.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "gemm_kernel.cuh"
#include "registry.h"

namespace {

using sat::GemmArgs;

template <int DT>
using ProbeTraits = sat::Traits<DT, 128, 1, sat::kProdTMA>;

template <int DT>
__global__ void __launch_bounds__(ProbeTraits<DT>::THREADS, 1)
    sat_gemm_relu_megakernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmC, const GemmArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    // Phase 1: this CTA's share of the GEMM.
    sat::gemm_cta<DT, 128, 1, sat::kProdTMA>(&tmA, tmB, tmC, args, smem_raw);
    // Phase 2: ReLU over the same tiles, in the order the schedule gave them.
    __syncthreads();
    sat::WorkIter it = sat::work_begin(args, blockIdx.x);
    sat::Unit w;
    while (sat::work_next(args, static_cast<int>(gridDim.x), it, w)) {
        const int r0 = w.tm * 128, c0 = w.tn * 128;
        for (int i = threadIdx.x; i < 128 * 128; i += blockDim.x) {
            const int r = r0 + i / 128, c = c0 + i % 128;
            if (r < args.M && c < args.N) {
                float* p = args.C + static_cast<int64_t>(r) * args.ldc + c;
                *p = fmaxf(*p, 0.0f);
            }
        }
    }
}

template <int DT>
cudaError_t launch_probe(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmC, const GemmArgs* a,
                         int grid, cudaStream_t stream)
{
    using T = ProbeTraits<DT>;
    cudaError_t e = cudaFuncSetAttribute(sat_gemm_relu_megakernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         T::SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    sat_gemm_relu_megakernel<DT><<<grid, T::THREADS, T::SMEM_BYTES, stream>>>(*tmA, *tmB, *tmC, *a);
    return cudaGetLastError();
}

}  // namespace

extern "C" int gemm_selftest_device_call(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, const void* A,
                                         const void* B, float* C, float alpha, float beta, void* cuda_stream)
{
    sat::set_last_error("");
    const int dt = static_cast<int>(dtype);
    if (M < 1 || N < 1 || K < 1 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31) ||
        dt < 0 || dt > 2)
        return sat::fail_with(GEMM_ERR_ARG, "bad dimensions or dtype");
    if (!A || !B || !C)
        return sat::fail_with(GEMM_ERR_ARG, "NULL operand");
    const int es = dt == 0 ? 4 : 2;
    if (reinterpret_cast<uintptr_t>(A) % 16 || reinterpret_cast<uintptr_t>(B) % 16 ||
        reinterpret_cast<uintptr_t>(C) % 16 || (K * es) % 16 || (N * es) % 16 || N % 4)
        return sat::fail_with(GEMM_ERR_ALIGN,
                              "the device-call self-test takes 16-byte aligned operands and row strides");
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return sat::fail_with(GEMM_ERR_LAUNCH, "querying the device: %s", cudaGetErrorString(e));

    const sat::KernelEntry* k = sat::find_entry(dt, 128, 1, sat::kProdTMA);
    if (!k)
        return sat::fail_with(GEMM_ERR_ARG, "no 128 x 128 kernel for this dtype");
    GemmArgs a{};
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.A = A;
    a.B = B;
    a.C = C;
    a.lda = static_cast<int>(K);
    a.ldb = static_cast<int>(N);
    a.ldc = static_cast<int>(N);
    a.alpha = alpha;
    a.beta = beta;
    a.tiles_m = static_cast<int>((M + 127) / 128);
    a.tiles_n = static_cast<int>((N + 127) / 128);
    a.num_kb = static_cast<int>((K + k->bk - 1) / k->bk);
    a.splits = 1;
    a.kb_per_split = a.num_kb;
    a.num_tiles = a.tiles_m * a.tiles_n;
    a.out_rows = static_cast<int>(M);
    a.group = 8;
    a.raster = 0;
    a.c_tma = 1;
    a.timeout_ns = 2000000000ull;

    const CUtensorMapDataType tdt = dt == 0   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                    : dt == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tmA{}, tmB{}, tmC{};
    if (sat::encode_map(&tmA, tdt, es, A, K, M, K, static_cast<uint32_t>(k->bk), 128u, CU_TENSOR_MAP_SWIZZLE_128B) ||
        sat::encode_map(&tmB, tdt, es, B, N, K, N, static_cast<uint32_t>(128 / es), static_cast<uint32_t>(k->bk),
                        static_cast<CUtensorMapSwizzle>(k->b_swizzle)) ||
        sat::encode_map(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, N, M, N, 32u, 32u, CU_TENSOR_MAP_SWIZZLE_128B))
        return sat::fail_with(GEMM_ERR_LAUNCH, "encoding the tensor maps");
    const int grid = static_cast<int>(a.num_tiles < sms ? a.num_tiles : sms);
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    e = dt == 0   ? launch_probe<0>(&tmA, &tmB, &tmC, &a, grid, stream)
        : dt == 1 ? launch_probe<1>(&tmA, &tmB, &tmC, &a, grid, stream)
                  : launch_probe<2>(&tmA, &tmB, &tmC, &a, grid, stream);
    if (e != cudaSuccess)
        return sat::fail_with(GEMM_ERR_LAUNCH, "launching the megakernel: %s", cudaGetErrorString(e));
    return GEMM_OK;
}
