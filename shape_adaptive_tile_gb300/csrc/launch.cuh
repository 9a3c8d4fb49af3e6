// Launcher and registry-entry builder for one kernel variant.
#pragma once

#include "gemm_kernel.cuh"
#include "registry.h"

namespace sat {

template <int DT, int BN, int CG, int PROD>
cudaError_t prepare_variant()
{
    using T = Traits<DT, BN, CG, PROD>;
    return cudaFuncSetAttribute(sat_gemm_kernel<DT, BN, CG, PROD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                T::SMEM_BYTES);
}

template <int DT, int BN, int CG, int PROD>
cudaError_t launch_variant(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmC,
                           const GemmArgs* args, int grid, cudaStream_t stream)
{
    using T = Traits<DT, BN, CG, PROD>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(T::THREADS, 1, 1);
    cfg.dynamicSmemBytes = T::SMEM_BYTES;
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
    return cudaLaunchKernelEx(&cfg, sat_gemm_kernel<DT, BN, CG, PROD>, *tmA, *tmB, *tmC, *args);
}

template <int DT, int BN, int CG, int PROD>
int max_clusters_variant()
{
    using T = Traits<DT, BN, CG, PROD>;
    if (CG != 2)
        return 0;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
    cfg.blockDim = dim3(T::THREADS, 1, 1);
    cfg.dynamicSmemBytes = T::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sat_gemm_kernel<DT, BN, CG, PROD>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

template <int DT, int BN, int CG, int PROD>
constexpr KernelEntry make_entry()
{
    using T = Traits<DT, BN, CG, PROD>;
    return KernelEntry{DT,
                       BN,
                       CG,
                       PROD,
                       T::STAGES,
                       T::THREADS,
                       T::SMEM_BYTES,
                       T::BK,
                       T::MN_LAYOUT == kLayoutSW128Atom32 ? static_cast<int>(CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B)
                                                         : static_cast<int>(CU_TENSOR_MAP_SWIZZLE_128B),
                       T::C_RING_OK ? 1 : 0,
                       T::A_MN ? 1 : 0,
                       T::B_KM ? 1 : 0,
                       &prepare_variant<DT, BN, CG, PROD>, &max_clusters_variant<DT, BN, CG, PROD>,
                       &launch_variant<DT, BN, CG, PROD>};
}

// The variants compiled for every dtype.
#define SAT_ENTRIES(DT)                                                                                         \
    make_entry<DT, 64, 1, kProdTMA>(), make_entry<DT, 128, 1, kProdTMA>(), make_entry<DT, 256, 1, kProdTMA>(), \
        make_entry<DT, 128, 2, kProdTMA>(), make_entry<DT, 256, 2, kProdTMA>(),                                 \
        make_entry<DT, 128, 1, kProdPlain>(), make_entry<DT, 256, 1, kProdPlain>(),                             \
        make_entry<DT, 128, 1, kProdPlainStrided>(), make_entry<DT, 256, 1, kProdPlainStrided>(),               \
        make_entry<DT, 32, 1, kProdSwap>(), make_entry<DT, 64, 1, kProdSwap>(), make_entry<DT, 128, 1, kProdSwap>(), \
        make_entry<DT, 128, 1, kProdTN>(), make_entry<DT, 256, 1, kProdTN>(), make_entry<DT, 256, 2, kProdTN>(),    \
        make_entry<DT, 128, 1, kProdNT>(), make_entry<DT, 256, 1, kProdNT>(), make_entry<DT, 256, 2, kProdNT>(),    \
        make_entry<DT, 128, 1, kProdTT>(), make_entry<DT, 256, 1, kProdTT>(), make_entry<DT, 256, 2, kProdTT>()

}  // namespace sat
