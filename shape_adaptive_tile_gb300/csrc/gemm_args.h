// Kernel arguments shared by the host launcher and the device code.
#pragma once

#include <cstdint>

namespace sat {

// Operand element types (same numbering as gemm_dtype_t in gemm.h).
constexpr int kDtTF32 = 0;
constexpr int kDtBF16 = 1;
constexpr int kDtFP16 = 2;

// Producer kinds.
constexpr int kProdTMA = 0;    // TMA tensor loads (16-byte aligned bases and strides)
constexpr int kProdPlain = 1;  // plain loads into the same swizzled layout (any stride)
constexpr int kProdSwap = 2;   // TMA loads, operand roles exchanged: the MMA computes C^T = B^T A^T
constexpr int kProdTN = 3;     // TMA loads, A stored transposed (K x M): first operand MN-major
constexpr int kProdNT = 4;     // TMA loads, B stored transposed (N x K): second operand K-major
constexpr int kProdTT = 5;     // TMA loads, both stored transposed
constexpr int kProdPlainStrided = 6;  // plain loads with row strides lda, ldb other than K, N
// TMA loads for rows that are not 16-byte aligned: A's rows are read through
// one tensor map per residue class of row index (rows m = r + P*y, whose
// byte offsets share one misalignment, aligned down), each output tile
// taking rows of one class; B is read from rows aligned in memory (the
// caller's, or an aligned copy), shifted in K by the class's offset.
constexpr int kProdClassA = 7;
constexpr int kMaxClasses = 8;

struct GemmArgs {
    int M, N, K;
    const void* A;             // M x K row-major (plain-load producer only)
    const void* B;             // K x N row-major (plain-load producer only)
    float* C;                  // output: C (M x N), or the split-K workspace (splits x out_rows x N)
    int lda, ldb;              // row strides of A and B in elements (plain-load producer only); < 2^31
    int ldc;                   // row stride of the output the kernel writes, in elements; < 2^31
    int c_half;                // element type of C: 0 fp32, 1 bf16, 2 fp16 (16-bit C: row-store epilogue only)
    float alpha, beta;
    int tiles_m, tiles_n;      // tiles of (128 * cta_group) x BN
    int num_tiles;             // work units: tiles_m * tiles_n * splits
    int num_kb;                // ceil(K / BK)
    int splits;                // K splits (1: C is written directly)
    int kb_per_split;          // k-blocks per split
    int out_rows;              // rows of one split's slice of the output (M, or the workspace's padded M)
    int group;                 // rasterisation group size (>= 1)
    int raster;                // 0: groups along M, 1: groups along N
    int c_tma;                 // 1: C is written (and read) through the TMA store path
    int c_ring;                // 1: the producer also fetches each tile's C (beta != 0) through the ring
    int alt_k;                 // 1: alternate waves of whole units run through K in opposite directions
    // Stream-K (sk_tiles > 0; only with splits == 1): the first sk_tiles tiles
    // in raster order are cut into k-block ranges of sk_w consecutive
    // positions of the (tile, k-block) sequence, one range per CTA slot
    // (CTA or CTA pair) g = 0 .. gridDim/cta_group - 1, taken before that
    // slot's whole tiles sk_tiles + g, sk_tiles + g + slots, ... A slot is
    // handed out by sk_ticket in the order the slots' CTAs start.
    int sk_tiles;
    int sk_w;
    float* sk_ws;              // per slot and CTA of a pair: 128 x BN fp32 partial tile
    unsigned* sk_flags;        // per slot and CTA of a pair: epilogue warps done with the partial
    unsigned* sk_ticket;       // slots handed out so far, over all launches on this scratch (may be null)
    unsigned sk_epoch;         // this launch's number (>= 1); a partial is ready at sk_epoch * epilogue warps
    // Class-view A (kProdClassA): P = a_classes residue classes of rows; class
    // r holds rows r + P*y, y < a_rows[r], read from a view that starts
    // a_shift[r] elements before each row (the aligned-down start). Output
    // tile rows tm = r + P*j: class r, view rows from j*128*cta_group.
    int a_classes;
    int a_rows[kMaxClasses];
    int a_shift[kMaxClasses];
    // Class-view tiles, fp32 C whose rows P apart lie a whole number of
    // 16-byte units apart (so all rows of a tile share one offset): the
    // epilogue stores the 16-byte-aligned part of each row in 16-byte units,
    // for rows that start on a 16-byte boundary (1) or for every row (2).
    int c_cls;
    uint32_t* err;             // device error word (bounded-wait timeouts), may be null
    unsigned long long timeout_ns;
};

}  // namespace sat
