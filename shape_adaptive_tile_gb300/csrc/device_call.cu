// The device-callable GEMM (include/gemm_device.cuh): gemm_device_prepare,
// which fills the routine's launch parameters, and gemm_selftest_device_call,
// a persistent kernel of the library's own built on the routine.
//
// "Measured data point on fixed-tile vs shape-adaptive GEMM" (section "The
// wall, and why we think it's structural") names the property a host API
// lacks: a GEMM that a persistent megakernel can call inline. The self-test
// kernel is the smallest such megakernel: phase 1 is the GEMM schedule of
// gemm_device_run; phase 2, in the same launch, applies max(x, 0) to the
// tiles of C that this CTA has just produced, reading them back from memory.
// Nothing between the phases is a launch boundary: the routine returns with
// its stores complete and ordered for the caller's generic accesses.
#include "gemm.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "gemm_device.cuh"
#include "registry.h"

namespace {

template <int DT, int BN, int CG>
__global__ void __launch_bounds__(GemmDeviceTile<DT, BN, CG>::THREADS, 1)
    sat_gemm_relu_megakernel(const __grid_constant__ gemm_device_params p)
{
    extern __shared__ uint8_t smem_raw[];
    // Phase 1: this CTA's share of the GEMM.
    gemm_device_run<DT, BN, CG>(p, smem_raw);
    // Phase 2: ReLU over the same tiles (this CTA's 128 rows of each), in the
    // order the schedule gave them.
    __syncthreads();
    const sat::GemmArgs& args = p.args;
    const int rank = CG == 2 ? static_cast<int>(sat::cluster_ctarank()) : 0;
    sat::WorkIter it = sat::work_begin(args, static_cast<int>(blockIdx.x) / CG);
    sat::Unit w;
    while (sat::work_next(args, static_cast<int>(gridDim.x) / CG, it, w)) {
        const int r0 = w.tm * 128 * CG + rank * 128, c0 = w.tn * BN;
        for (int i = threadIdx.x; i < 128 * BN; i += blockDim.x) {
            const int r = r0 + i / BN, c = c0 + i % BN;
            if (r < args.M && c < args.N) {
                float* q = args.C + static_cast<int64_t>(r) * args.ldc + c;
                *q = fmaxf(*q, 0.0f);
            }
        }
    }
}

template <int DT, int BN, int CG>
cudaError_t launch_selftest(const gemm_device_params& p, cudaStream_t stream)
{
    cudaError_t e = cudaFuncSetAttribute(sat_gemm_relu_megakernel<DT, BN, CG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(p.threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(p.smem_bytes);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (CG == 2) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, sat_gemm_relu_megakernel<DT, BN, CG>, p);
}

}  // namespace

extern "C" int gemm_device_prepare(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, const void* A, const void* B,
                                   float* C, float alpha, float beta, int cta_group, void* params,
                                   int64_t params_bytes)
{
    sat::set_last_error("");
    const int dt = static_cast<int>(dtype);
    if (M < 1 || N < 1 || K < 1 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31) ||
        dt < 0 || dt > 2 || (cta_group != 1 && cta_group != 2))
        return sat::fail_with(GEMM_ERR_ARG, "bad dimensions, dtype or cta_group");
    if (!A || !B || !C || !params || params_bytes < static_cast<int64_t>(sizeof(gemm_device_params)))
        return sat::fail_with(GEMM_ERR_ARG, "NULL operand, or params smaller than gemm_device_params (%zu bytes)",
                              sizeof(gemm_device_params));
    if (reinterpret_cast<uintptr_t>(params) % 64)
        return sat::fail_with(GEMM_ERR_ALIGN, "params must be 64-byte aligned (it holds tensor maps)");
    const int es = dt == 0 ? 4 : 2;
    if (reinterpret_cast<uintptr_t>(A) % 16 || reinterpret_cast<uintptr_t>(B) % 16 ||
        reinterpret_cast<uintptr_t>(C) % 16 || (K * es) % 16 || (N * es) % 16 || N % 4)
        return sat::fail_with(GEMM_ERR_ALIGN, "the device routine takes 16-byte aligned operands and row strides");
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return sat::fail_with(GEMM_ERR_LAUNCH, "querying the device: %s", cudaGetErrorString(e));

    const int bn = cta_group == 2 ? 256 : 128;
    const sat::KernelEntry* k = sat::find_entry(dt, bn, cta_group, sat::kProdTMA);
    if (!k)
        return sat::fail_with(GEMM_ERR_ARG, "no compiled tile for cta_group %d", cta_group);
    gemm_device_params p{};
    sat::GemmArgs& a = p.args;
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
    a.tiles_m = static_cast<int>((M + 128 * cta_group - 1) / (128 * cta_group));
    a.tiles_n = static_cast<int>((N + bn - 1) / bn);
    a.num_kb = static_cast<int>((K + k->bk - 1) / k->bk);
    a.splits = 1;
    a.kb_per_split = a.num_kb;
    a.num_tiles = a.tiles_m * a.tiles_n;
    a.out_rows = static_cast<int>(M);
    a.group = 8;
    a.raster = 0;
    a.alt_k = 1;
    a.c_tma = 1;
    a.timeout_ns = 2000000000ull;

    const CUtensorMapDataType tdt = dt == 0   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                    : dt == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (sat::encode_map(&p.tmA, tdt, es, A, K, M, K, static_cast<uint32_t>(k->bk), 128u, CU_TENSOR_MAP_SWIZZLE_128B) ||
        sat::encode_map(&p.tmB, tdt, es, B, N, K, N, static_cast<uint32_t>(128 / es), static_cast<uint32_t>(k->bk),
                        static_cast<CUtensorMapSwizzle>(k->b_swizzle)) ||
        sat::encode_map(&p.tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, N, M, N, 32u, 32u, CU_TENSOR_MAP_SWIZZLE_128B))
        return sat::fail_with(GEMM_ERR_LAUNCH, "encoding the tensor maps");
    // Blocks: one per tile, at most the co-resident blocks (pairs: as many as
    // the occupancy calculator fits).
    int64_t slots = sms / cta_group;
    if (cta_group == 2) {
        const int n = k->max_clusters();
        if (n > 0 && n < slots)
            slots = n;
    }
    p.threads = k->threads;
    p.smem_bytes = k->smem;
    p.cluster_size = cta_group;
    p.grid = static_cast<int>((a.num_tiles < slots ? a.num_tiles : slots) * cta_group);
    p.bn = bn;
    p.cta_group = cta_group;
    *static_cast<gemm_device_params*>(params) = p;
    return GEMM_OK;
}

extern "C" int gemm_selftest_device_call(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, const void* A,
                                         const void* B, float* C, float alpha, float beta, int cta_group,
                                         void* cuda_stream)
{
    alignas(64) gemm_device_params p;
    const int rc = gemm_device_prepare(M, N, K, dtype, A, B, C, alpha, beta, cta_group, &p, sizeof p);
    if (rc)
        return rc;
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    const int dt = static_cast<int>(dtype);
    cudaError_t e;
    if (cta_group == 2)
        e = dt == 0 ? launch_selftest<0, 256, 2>(p, stream)
            : dt == 1 ? launch_selftest<1, 256, 2>(p, stream)
                      : launch_selftest<2, 256, 2>(p, stream);
    else
        e = dt == 0 ? launch_selftest<0, 128, 1>(p, stream)
            : dt == 1 ? launch_selftest<1, 128, 1>(p, stream)
                      : launch_selftest<2, 128, 1>(p, stream);
    if (e != cudaSuccess)
        return sat::fail_with(GEMM_ERR_LAUNCH, "launching the megakernel: %s", cudaGetErrorString(e));
    return GEMM_OK;
}
