/*
 * The GEMM as a device routine, for persistent kernels of the caller's own.
 *
 * "Measured data point on fixed-tile vs shape-adaptive GEMM" (section "What
 * we measured") singles out what a host API cannot offer: a GEMM callable
 * inline from a persistent megakernel. This header is that form of the
 * library's kernel: gemm_device_run() is the whole persistent GEMM schedule
 * of one CTA (TMA ring, tcgen05.mma into tensor memory, double-buffered
 * accumulators, epilogue), callable as one phase of a longer kernel, with
 * other work before or after it in the same launch.
 *
 * Use, in CUDA C++ compiled for sm_103a (nvcc -gencode
 * arch=compute_103a,code=sm_103a, with this directory and the library's
 * csrc/ directory on the include path):
 *
 *   1. On the host, fill a gemm_device_params with gemm_device_prepare()
 *      (include/gemm.h): tensor maps of A, B and C, the schedule, and the
 *      launch shape it needs (threads, dynamic shared memory, cluster size,
 *      grid).
 *   2. Launch a kernel of yours with exactly params.threads threads per
 *      block, params.smem_bytes of dynamic shared memory (after
 *      cudaFuncSetAttribute(..., cudaFuncAttributeMaxDynamicSharedMemorySize,
 *      ...)), params.grid blocks in clusters of params.cluster_size, and the
 *      params as a __grid_constant__ parameter.
 *   3. In it, let every thread of every block call
 *      gemm_device_run<DTYPE, BN, CG>(params, smem) once, DTYPE/BN/CG being
 *      the instance gemm_device_prepare() named (GEMM_DEVICE_TILE below).
 *
 * Conditions (they are the routine's; breaking one hangs until the bounded
 * waits give up, or gives a wrong C):
 *   - every block of the grid calls the routine, with all of its threads;
 *   - no other use of the dynamic shared memory overlaps the call;
 *   - the tensor memory of the SM is free while the call runs (the routine
 *     allocates its accumulators there and frees them before returning).
 * On return, the block's share of C is written, its bulk stores are
 * complete and made visible to the block's later generic loads, and its
 * tensor memory is freed: the caller may read the block's tiles back
 * (sat::work_begin / sat::work_next give which ones, in schedule order).
 * Reading other blocks' tiles needs a grid-wide synchronisation first.
 */
#ifndef SAT_GEMM_DEVICE_CUH
#define SAT_GEMM_DEVICE_CUH

#include <cuda.h>
#include <stdint.h>

#include "gemm.h"
#include "gemm_kernel.cuh"

/* Launch shape and arguments of the device routine, as gemm_device_prepare()
 * fills them. Tensor maps first (each needs 64-byte alignment). */
struct gemm_device_params {
    CUtensorMap tmA, tmB, tmC;
    sat::GemmArgs args;
    int threads;       /* threads per block */
    int smem_bytes;    /* dynamic shared memory per block */
    int cluster_size;  /* 1, or 2 for CTA pairs (launch in clusters of 2) */
    int grid;          /* blocks: the tiles, at most the co-resident blocks */
    int bn;            /* the instance: tile N (128 for cta_group 1, 256 for 2) */
    int cta_group;     /* the instance: 1 or 2 */
};

/* The instances gemm_device_prepare() names: (bn, cta_group) = (128, 1) or
 * (256, 2), with TMA loads and the deepest ring. */
template <int DT, int BN, int CG>
struct GemmDeviceTile {
    using T = sat::Traits<DT, BN, CG, sat::kProdTMA>;
    static constexpr int THREADS = T::THREADS;
    static constexpr int SMEM_BYTES = T::SMEM_BYTES;
};

/* The GEMM phase: this block's share of C = alpha * A * B + beta * C. */
template <int DT, int BN, int CG>
__device__ __forceinline__ void gemm_device_run(const gemm_device_params& p, uint8_t* smem)
{
    sat::gemm_cta<DT, BN, CG, sat::kProdTMA>(&p.tmA, p.tmB, p.tmC, p.args, smem);
}

#endif /* SAT_GEMM_DEVICE_CUH */
