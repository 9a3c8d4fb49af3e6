// The shape-adaptive dispatcher: (M, N, K, dtype, SM count) -> kernel choice.
#pragma once

#include <cstdint>

namespace sat {

struct Choice {
    int bn;       // tile N
    int cg;       // 1 or 2 (CTA pair)
    int raster;   // 0: groups along M, 1: groups along N
    int group;    // raster group size in tiles
    int source;   // 0: analytic rule, 1: committed sweep table, 2: forced
    int splits;   // K splits (fixed-order reduction through a workspace); 0 or 1: none
    int cload;    // beta != 0: 1 = the epilogue loads C itself, 0 = the producer fetches it through the ring
    int sk;       // 1: stream-K for the last waves of tiles (fixed-order fix-up of split tiles)
    int swap;     // 1: operand roles exchanged (the MMA computes C^T = B^T A^T; bn tiles M), 1-SM only
    int stages;   // shared-memory ring depth of the TMA kernel; 0: the deepest compiled for the tile
};

// Source codes of a choice.
constexpr int kSrcRule = 0, kSrcTable = 1, kSrcForced = 2, kSrcBucket = 3;

// Estimated DRAM bytes that reading the operands takes when `tiles_m` x
// `tiles_n` output tiles (rows of `tile_rows` of A, columns of `tile_cols` of
// B, each needing its whole K panel of `row_bytes` per row or column) run in
// raster order (raster, group) as waves of `slots` concurrent tiles, with
// the first `lead` tiles as one wave of their own (stream-K pieces). L2 is a
// least-recently-used store of whole panels of `l2_bytes`.
double operand_traffic(int64_t tiles_m, int64_t tiles_n, int64_t tile_rows, int64_t tile_cols, double row_bytes,
                       int raster, int group, int64_t slots, int64_t lead, double l2_bytes);

// Stream-K layout for T output tiles of KB k-blocks on G CTA slots: the
// first *sk_tiles tiles (in raster order) are shared out as ranges of *sk_w
// consecutive (tile, k-block) positions, one range per slot, which each
// slot runs before its whole tiles. The shared tiles are those of the
// partial last wave, or, where that would cut a tile into more than about
// five pieces, those of the last full wave too. Returns false (no
// stream-K) with at most one wave of tiles (measured slower there), when
// the tiles fill whole waves exactly, or when the positions would not fit
// an int.
bool sk_layout(int64_t T, int64_t KB, int64_t G, int* sk_tiles, int* sk_w);

// Picks tile and schedule. `tma_ok` says whether the TMA load path can be
// used (16-byte-multiple row strides); when false only 1-SM tiles exist.
Choice select_config(int64_t M, int64_t N, int64_t K, int dt, int sm_count, bool tma_ok);

// Override for sweeps and tests: "bn,cg,raster,group[,splits]" (e.g. "256,2,0,8");
// tags such as ",cload" are stripped by the caller first.
// Returns false if `spec` is malformed.
bool parse_choice(const char* spec, Choice* out);

}  // namespace sat
