// Table of compiled kernel variants, one entry per (dtype, BN, cta_group,
// producer). The dispatcher picks among these; the launcher runs one.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_args.h"

namespace sat {

struct KernelEntry {
    int dt;        // kDtTF32 / kDtBF16 / kDtFP16
    int bn;        // N of the output tile
    int cg;        // 1: one SM per 128-row tile; 2: a CTA pair (cluster of 2) per 256-row tile
    int prod;      // kProdTMA, kProdPlain, kProdSwap, kProdTN/NT/TT or kProdPlainStrided
    int stages;    // shared-memory ring depth
    int threads;   // CTA size
    int smem;      // dynamic shared memory bytes
    int bk;        // K per stage
    int b_swizzle; // CUtensorMapSwizzle of MN-major operand boxes (B as it lies, or A stored K x M)
    int c_ring;    // 1: with beta != 0 the producer can fetch C through the operand ring
    int a_mn;      // 1: the first MMA operand is read MN-major (A stored K x M, or B for a swapped tile)
    int b_km;      // 1: the second MMA operand is read K-major (B stored N x K, or A for a swapped tile)
    cudaError_t (*prepare)();  // sets the kernel's dynamic shared-memory limit
    int (*max_clusters)();     // co-resident CTA pairs on this device (cg == 2), 0 if unknown
    cudaError_t (*launch)(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmC,
                          const GemmArgs* args, int grid, cudaStream_t stream);
};

// Defined in kernels_<dtype>.cu, kernels_<dtype>_alt.cu and kernels_<dtype>_trans.cu.
extern const KernelEntry kEntriesTF32[], kEntriesTF32Alt[], kEntriesTF32Trans[];
extern const int kNumEntriesTF32, kNumEntriesTF32Alt, kNumEntriesTF32Trans;
extern const KernelEntry kEntriesBF16[], kEntriesBF16Alt[], kEntriesBF16Trans[];
extern const int kNumEntriesBF16, kNumEntriesBF16Alt, kNumEntriesBF16Trans;
extern const KernelEntry kEntriesFP16[], kEntriesFP16Alt[], kEntriesFP16Trans[];
extern const int kNumEntriesFP16, kNumEntriesFP16Alt, kNumEntriesFP16Trans;

// Sets the message gemm_last_error() returns on this thread (api.cu).
void set_last_error(const char* msg);

// Sets that message from a printf format and returns `code` (api.cu).
int fail_with(int code, const char* fmt, ...);

// Encodes a 2-D tensor map of a row-major matrix: `outer` rows of `inner`
// elements, `ld` elements apart, read or written in boxes of box_inner x
// box_outer with the given swizzle and zero fill outside the matrix.
// Returns 0, -1 if the driver's encoder is unavailable, or the driver's
// error code (tensor_map.cpp).
int encode_map(CUtensorMap* map, CUtensorMapDataType type, int elem_bytes, const void* ptr, uint64_t inner,
               uint64_t outer, uint64_t ld, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);

// Finds the variant with `stages` ring stages (0: the deepest ring compiled
// for that tile), or nullptr.
const KernelEntry* find_entry(int dt, int bn, int cg, int prod, int stages = 0);

// The output tiles of a variant, as rows of tiles (the accumulator's 128 x
// cta_group rows) and columns of tiles (its bn columns). A swapped variant
// tiles C^T: 128 columns of C by bn rows.
inline void tile_grid(const KernelEntry* e, int64_t M, int64_t N, int64_t* tiles_m, int64_t* tiles_n)
{
    const int64_t rows = e->prod == kProdSwap ? N : M, cols = e->prod == kProdSwap ? M : N;
    *tiles_m = (rows + 128 * e->cg - 1) / (128 * e->cg);
    *tiles_n = (cols + e->bn - 1) / e->bn;
}

// Defined in aux_kernels.cu. C is rows x cols elements with row stride ldc,
// of kind 0 (fp32), 1 (bf16) or 2 (fp16).
cudaError_t launch_scale(float* C, int kind, long long rows, long long cols, long long ldc, float beta,
                         cudaStream_t stream);
cudaError_t launch_wait_probe(uint32_t* err, unsigned long long timeout_ns, cudaStream_t stream);
cudaError_t launch_pack_rows(const void* src, long long ld_src_bytes, void* dst, long long ld_dst_bytes,
                             long long rows, long long row_bytes, int sm_count, cudaStream_t stream);
cudaError_t launch_splitk_reduce(const float* ws, int S, long long slice, float* C, int kind, long long rows,
                                 long long cols, long long ldc, float alpha, float beta, int sm_count,
                                 cudaStream_t stream);

}  // namespace sat
