// Launcher and registry-entry builder for one kernel variant.
#pragma once

#include "gemm_kernel.cuh"
#include "registry.h"

namespace sat {

// The kernel of a variant: class-view A takes one tensor map per class.
template <int DT, int BN, int CG, int PROD, int ST>
constexpr auto kernel_of()
{
    if constexpr (PROD == kProdClassA)
        return sat_gemm_cls_kernel<DT, BN, CG, ST>;
    else
        return sat_gemm_kernel<DT, BN, CG, PROD, ST>;
}

template <int DT, int BN, int CG, int PROD, int ST>
cudaError_t prepare_variant()
{
    using T = Traits<DT, BN, CG, PROD, ST>;
    return cudaFuncSetAttribute(kernel_of<DT, BN, CG, PROD, ST>(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                T::SMEM_BYTES);
}

template <int DT, int BN, int CG, int PROD, int ST>
cudaError_t launch_variant(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmC,
                           const GemmArgs* args, int grid, cudaStream_t stream)
{
    using T = Traits<DT, BN, CG, PROD, ST>;
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
    if constexpr (PROD == kProdClassA) {
        // tmA points to args->a_classes maps, one per residue class of row index.
        ClassMaps maps{};
        for (int i = 0; i < args->a_classes && i < kMaxClasses; ++i)
            maps.a[i] = tmA[i];
        return cudaLaunchKernelEx(&cfg, sat_gemm_cls_kernel<DT, BN, CG, ST>, maps, *tmB, *tmC, *args);
    } else {
        return cudaLaunchKernelEx(&cfg, sat_gemm_kernel<DT, BN, CG, PROD, ST>, *tmA, *tmB, *tmC, *args);
    }
}

template <int DT, int BN, int CG, int PROD, int ST>
int max_clusters_variant()
{
    using T = Traits<DT, BN, CG, PROD, ST>;
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
    if (cudaOccupancyMaxActiveClusters(&n, kernel_of<DT, BN, CG, PROD, ST>(), &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

template <int DT, int BN, int CG, int PROD, int ST>
constexpr KernelEntry make_entry()
{
    using T = Traits<DT, BN, CG, PROD, ST>;
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
                       &prepare_variant<DT, BN, CG, PROD, ST>, &max_clusters_variant<DT, BN, CG, PROD, ST>,
                       &launch_variant<DT, BN, CG, PROD, ST>};
}

// The variants compiled for every dtype, in three groups (one translation
// unit each, so that they compile in parallel).
// Untransposed TMA tiles, with two ring depths each: the most stages that
// fit, and a shallower ring (a dispatcher dimension, measured by the sweep).
#define SAT_ENTRIES_TMA(DT)                                                                                     \
    make_entry<DT, 64, 1, kProdTMA, 0>(), make_entry<DT, 128, 1, kProdTMA, 0>(),                                \
        make_entry<DT, 256, 1, kProdTMA, 0>(), make_entry<DT, 128, 2, kProdTMA, 0>(),                           \
        make_entry<DT, 256, 2, kProdTMA, 0>(), make_entry<DT, 64, 1, kProdTMA, 4>(),                            \
        make_entry<DT, 128, 1, kProdTMA, 4>(), make_entry<DT, 256, 1, kProdTMA, 3>(),                           \
        make_entry<DT, 128, 2, kProdTMA, 4>(), make_entry<DT, 256, 2, kProdTMA, 4>()
// Plain loads, swapped operands and class views of A.
#define SAT_ENTRIES_ALT(DT)                                                                                     \
    make_entry<DT, 128, 1, kProdPlain, 0>(), make_entry<DT, 256, 1, kProdPlain, 0>(),                           \
        make_entry<DT, 128, 1, kProdPlainStrided, 0>(), make_entry<DT, 256, 1, kProdPlainStrided, 0>(),         \
        make_entry<DT, 32, 1, kProdSwap, 0>(), make_entry<DT, 64, 1, kProdSwap, 0>(),                           \
        make_entry<DT, 128, 1, kProdSwap, 0>(), make_entry<DT, 128, 1, kProdClassA, 0>(),                       \
        make_entry<DT, 256, 1, kProdClassA, 0>(), make_entry<DT, 256, 2, kProdClassA, 0>()
// Transposed operands.
#define SAT_ENTRIES_TRANS(DT)                                                                                   \
    make_entry<DT, 128, 1, kProdTN, 0>(), make_entry<DT, 256, 1, kProdTN, 0>(),                                 \
        make_entry<DT, 256, 2, kProdTN, 0>(), make_entry<DT, 128, 1, kProdNT, 0>(),                             \
        make_entry<DT, 256, 1, kProdNT, 0>(), make_entry<DT, 256, 2, kProdNT, 0>(),                             \
        make_entry<DT, 128, 1, kProdTT, 0>(), make_entry<DT, 256, 1, kProdTT, 0>(),                             \
        make_entry<DT, 256, 2, kProdTT, 0>()

}  // namespace sat
