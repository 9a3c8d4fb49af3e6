// Persistent, warp-specialised tcgen05 GEMM for sm_103a:
//     C[M x N] = alpha * A[M x K] * B[K x N] + beta * C      (row-major, fp32 C)
//
// This is the fixed-schedule kernel that "Measured data point on fixed-tile
// vs shape-adaptive GEMM" (section "The wall, and why we think it's
// structural") says is not enough on its own, re-done for Blackwell: every
// instantiation is one (tile, schedule) point among which the shape-adaptive
// dispatcher chooses.
//
// Roles (one CTA per SM, or a CTA pair on two SMs for cta_group::2):
//   producer warp(s): fill an S-stage shared-memory ring, by TMA (2-D tiled
//       loads, 128-byte swizzle, zero fill outside the matrix) or, when a row
//       stride is not a multiple of 16 bytes, by plain loads written into the
//       same swizzled layout;
//   MMA warp: one thread issues tcgen05.mma (kind::tf32 or kind::f16) from
//       the ring into a TMEM accumulator, releasing each stage with
//       tcgen05.commit; two accumulators alternate so that the epilogue of one
//       tile overlaps the main loop of the next;
//   4 epilogue warps: tcgen05.ld TMEM -> registers, transpose through a
//       per-warp shared buffer, then alpha*acc (+ beta*C) with row-contiguous,
//       masked stores (no alignment needed, any M/N tail).
// The K loop always runs k = 0..K-1 in the same order for a tile, and no
// output element is produced by more than one CTA, so results are
// bit-identical from run to run.
#pragma once

#include <cstdint>
#include <type_traits>
#include <cuda.h>

#include "gemm_args.h"
#include "ptx.cuh"

namespace sat {

// Error bits written to the device error word.
constexpr uint32_t kErrTimeoutProducer = 1u << 0;
constexpr uint32_t kErrTimeoutMma = 1u << 1;
constexpr uint32_t kErrTimeoutEpilogue = 1u << 2;
constexpr uint32_t kErrTimeoutDrain = 1u << 3;
constexpr uint32_t kErrTimeoutPartial = 1u << 4;   // a stream-K partial tile never arrived
constexpr uint32_t kErrTicket = 1u << 5;           // a stream-K slot ticket outside this launch's range

// ST: shared-memory ring depth, 0 for the most stages that fit.
template <int DT, int BN, int CG, int PROD, int ST = 0>
struct Traits {
    static constexpr bool PLAIN = PROD == kProdPlain || PROD == kProdPlainStrided;  // plain-load producer warps
    static constexpr bool TMA = !PLAIN;  // one elected thread issues TMA loads
    // Operand roles exchanged: the tensor core computes C^T = B^T A^T, its
    // 128 accumulator rows being 128 columns n of C and its BN columns BN
    // rows m of C. The first MMA operand is B^T, read from B as it lies
    // (n contiguous, MN-major); the second is A^T, read from A as it lies (k
    // contiguous, K-major). For skinny M, where 128-row tiles of C would be
    // mostly empty.
    static constexpr bool SWAP = PROD == kProdSwap;
    // Class-view A (rows whose byte offsets are not 16-byte aligned): one
    // tensor map per residue class of row index, and a fixer warp that zeroes
    // the elements of the previous row that each tile's first k-block reads
    // in front of every row (the views start aligned down).
    static constexpr bool CLS = PROD == kProdClassA;
    // Operand layouts in shared memory: the first MMA operand (the
    // accumulator's rows) MN-major when it comes from a matrix stored with
    // those rows contiguous (A stored K x M, or B for a swapped tile), else
    // K-major; the second (its columns) K-major when it comes from a matrix
    // stored with K contiguous (B stored N x K, or A for a swapped tile),
    // else MN-major.
    static constexpr bool A_MN = SWAP || PROD == kProdTN || PROD == kProdTT;
    static constexpr bool B_KM = SWAP || PROD == kProdNT || PROD == kProdTT;
    static constexpr bool kTF32 = DT == kDtTF32;
    static constexpr int ES = kTF32 ? 4 : 2;        // bytes per operand element
    static constexpr int BM = 128;                  // accumulator rows per CTA
    static constexpr int BK = 128 / ES;             // one 128-byte swizzle row of K
    static constexpr int UK = 32 / ES;              // K of one MMA instruction
    static constexpr int KSTEPS = BK / UK;
    static constexpr int CW = 128 / ES;             // B columns per swizzle row
    static constexpr int BN_CTA = BN / CG;          // B columns this CTA loads
    static constexpr int NBOX = BN_CTA / CW;        // B boxes per stage
    static constexpr int A_BYTES = BM * 128;
    static constexpr int NBOX_A = BM / CW;          // MN-major first operand: boxes of CW rows per stage
    static constexpr int B_BYTES = BN_CTA * 128;    // either layout: BN_CTA x BK elements
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // Epilogue: 8 warps (4 with the plain-load producer), two (one) per TMEM
    // lane quarter, taking alternate 32-column chunks. Each has one 4 KB staging buffer: 32 rows x 128
    // bytes in the TMA store's 128-byte swizzle for the bulk-store path, or
    // a 32 x 32 XOR-swizzled transpose buffer for the row-store fallback.
    static constexpr int EPI_WARPS = TMA ? 8 : 4;   // plain-load CTAs keep 9 warps
    static constexpr int EPI_WARP_BYTES = 4096;
    static constexpr int EPI_BYTES = EPI_WARPS * EPI_WARP_BYTES;
    static constexpr int BAR_BYTES = 512;
    static constexpr int BUDGET = 227 * 1024 - 1024 - EPI_BYTES - BAR_BYTES;
    static constexpr int MAX_STAGES = (BUDGET / STAGE_BYTES) > 8 ? 8 : (BUDGET / STAGE_BYTES);
    static constexpr int STAGES = ST > 0 && ST < MAX_STAGES ? ST : MAX_STAGES;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
    static constexpr int NPW = TMA ? 1 : 4;   // producer warps
    static constexpr int MMA_WARP = NPW;
    static constexpr int EPI_WARP0 = NPW + 1;
    static constexpr int FIX_WARP = CLS ? EPI_WARP0 + EPI_WARPS : -1;
    static constexpr int THREADS = (NPW + 1 + EPI_WARPS + (CLS ? 1 : 0)) * 32;
    static constexpr int ACC_COLS = BN;             // fp32 accumulator: one column per element
    // beta != 0: the producer can fetch each tile's C (this CTA's BM x BN
    // fp32 block, as 32 x 32 chunks of 4 KB in the 128-byte swizzle) through
    // the operand ring, right after the tile's k-blocks: CPS chunks per
    // stage, NCS stages per tile, at least two stages left for k-blocks.
    static constexpr int C_CHUNKS = (BM / 32) * (BN / 32);
    static constexpr int CPS = STAGE_BYTES / 4096;
    static constexpr int NCS = (C_CHUNKS + CPS - 1) / CPS;
    static constexpr bool C_RING_OK = PROD == kProdTMA && NCS + 2 <= STAGES;
    static constexpr int TMEM_COLS = 2 * BN <= 64 ? 64 : 2 * BN <= 128 ? 128 : 2 * BN <= 256 ? 256 : 512;
    static constexpr uint32_t FMT = DT == kDtTF32 ? kFmtTF32 : DT == kDtBF16 ? kFmtBF16 : kFmtF16;
    // Operand tiles in shared memory, each as it lies in memory.
    // MN-major (M or N contiguous): 16-bit types in the 128-byte swizzle,
    // 32-bit (tf32) types in the 128-byte swizzle with 32-byte atoms, the only
    // MN-major swizzle the tensor core takes for 32-bit operands; 128-byte
    // column blocks are BK*128 bytes apart (leading byte offset); K rows come
    // in swizzle groups, 8 rows (1024 bytes) for 16-byte atoms and 4 rows (512
    // bytes) for 32-byte atoms (stride byte offset); one MMA step of K advances
    // UK rows of 128 bytes. K-major: rows of 128 bytes in the 128-byte swizzle,
    // 8-row groups 1024 bytes apart; one MMA step of K advances 32 bytes
    // inside the swizzled row. The plain-load producers write the same
    // layouts (B MN-major) themselves.
    static constexpr uint32_t IDESC = idesc_f32acc(FMT, BM * CG, BN, !B_KM, A_MN);
    static constexpr uint32_t MN_LAYOUT = kTF32 ? kLayoutSW128Atom32 : kLayoutSW128;
    static constexpr uint32_t MN_LBO = BK * 128;
    static constexpr uint32_t MN_SBO = MN_LAYOUT == kLayoutSW128Atom32 ? 512 : 1024;
    static constexpr uint32_t MN_KSTEP = UK * 128;
    static constexpr uint32_t K_KSTEP = UK * ES;     // = 32

    static_assert(B_KM || BN % (CW * CG) == 0, "B tile must be whole swizzle rows per CTA");
    static_assert(!B_KM || BN_CTA % 8 == 0, "K-major tile: whole 8-row swizzle groups");
    static_assert(BK == CW, "one 128-byte row of K per stage");
    static_assert(!SWAP || (CG == 1 && BN >= 32), "swapped tiles: 1-SM, whole 32-column chunks");
    static_assert(BN >= 16 && BN <= 256 && BN % 16 == 0, "MMA N");
    static_assert(STAGES >= 2, "ring too small");
    static_assert(!PLAIN || CG == 1, "plain-load producer is 1-SM only");
    static_assert(2 * BN <= 512, "two accumulators must fit in TMEM");
};

__device__ __forceinline__ void tile_coord(int t, const GemmArgs& a, int& tm, int& tn)
{
    if (a.raster == 0) {  // groups of `group` tile-rows, rows fastest inside a group
        const int per = a.group * a.tiles_n;
        const int g = t / per, r = t - g * per;
        const int first = g * a.group;
        const int gs = min(a.group, a.tiles_m - first);
        tm = first + r % gs;
        tn = r / gs;
    } else {              // groups of `group` tile-columns, columns fastest
        const int per = a.group * a.tiles_m;
        const int g = t / per, r = t - g * per;
        const int first = g * a.group;
        const int gs = min(a.group, a.tiles_n - first);
        tn = first + r % gs;
        tm = r / gs;
    }
}

// Byte offset of operand element (row r, k) in a K-major 128-byte-swizzled
// tile: 16-byte chunk index XOR (row mod 8), rows 128 bytes apart.
template <int ES>
__device__ __forceinline__ uint32_t swz_kmajor(int r, int k)
{
    const uint32_t kb = static_cast<uint32_t>(k * ES);
    return static_cast<uint32_t>(r) * 128u + ((((kb >> 4) ^ static_cast<uint32_t>(r & 7)) << 4) | (kb & 15u));
}

// A work unit: output tile (tm, tn) of K split s, k-blocks [kb0, kb1).
// Units of one split are consecutive, so CTAs running at the same time
// share that split's K slice of the operands in L2.
//
// Stream-K pieces come in three kinds: a whole tile; a partial piece (it
// ends before the tile's last k-block), whose raw sum goes to its slot's
// partial tile; and a final piece (k-blocks kb0 > 0 .. num_kb), which adds
// the partial pieces of slots first .. g - 1, in that order, before the
// epilogue. A final piece thus waits only on slots that started before its
// own, and only on each one's first unit.
constexpr int kWhole = 0, kSkPartial = 1, kSkFinal = 2;

// rev: the unit runs its k-blocks from kb1 - 1 down to kb0 (see work_next).
struct Unit {
    int tm, tn, s, kb0, kb1, kind, first, rev;
};

__device__ __forceinline__ Unit unit_coord(int u, const GemmArgs& a)
{
    Unit w;
    const int per = a.tiles_m * a.tiles_n;
    w.s = u / per;
    tile_coord(u - w.s * per, a, w.tm, w.tn);
    w.kb0 = w.s * a.kb_per_split;
    w.kb1 = min(a.num_kb, w.kb0 + a.kb_per_split);
    w.kind = kWhole;
    w.first = 0;
    w.rev = 0;
    return w;
}

// The sequence of units of CTA slot g out of G: its stream-K range of
// (tile, k-block) positions [pos, end), cut at tile boundaries and taken
// from the end backwards, then its whole units t = sk_tiles + g,
// sk_tiles + g + G, ... Without stream-K this is t = g, g + G, ...
//
// Taken backwards, a range's first unit is the piece that starts the last
// tile it touches (or, inside one tile, the whole range): a partial piece,
// or a whole tile, that waits on nobody. Its last unit is the piece that
// ends the first tile it touches, the tile's final piece, which waits for
// the pieces of the slots before it: each is that slot's first unit.
struct WorkIter {
    int pos, end, t;
};

__device__ __forceinline__ WorkIter work_begin(const GemmArgs& a, int g)
{
    WorkIter it;
    const int total = a.sk_tiles * a.num_kb;
    it.pos = a.sk_tiles > 0 ? min(g * a.sk_w, total) : 0;
    it.end = a.sk_tiles > 0 ? min(it.pos + a.sk_w, total) : 0;
    it.t = a.sk_tiles + g;
    return it;
}

template <bool kSK = true>
__device__ __forceinline__ bool work_next(const GemmArgs& a, int G, WorkIter& it, Unit& w)
{
    if (kSK && it.pos < it.end) {
        const int tile = (it.end - 1) / a.num_kb;
        const int tstart = tile * a.num_kb;
        const int p0 = max(it.pos, tstart);
        tile_coord(tile, a, w.tm, w.tn);
        w.s = 0;
        w.kb0 = p0 - tstart;
        w.kb1 = it.end - tstart;
        w.kind = w.kb1 < a.num_kb ? kSkPartial : (w.kb0 > 0 ? kSkFinal : kWhole);
        w.first = tstart / a.sk_w;   // the slot whose range holds the tile's k-block 0
        w.rev = 0;
        it.end = p0;
        return true;
    }
    if (it.t < a.num_tiles) {
        w = unit_coord(it.t, a);
        // Alternate waves of whole units run through K in opposite directions
        // (a.alt_k): a wave whose panels exceed L2 leaves the last k-blocks
        // it read there, which the next wave, reversed, reads first. After
        // stream-K pieces (which end on tiles' last k-blocks) the first wave
        // is a reversed one. The order depends only on the layout, so it is
        // the same on every run.
        w.rev = a.alt_k ? (((it.t - a.sk_tiles) / G) + (a.sk_tiles > 0 ? 1 : 0)) & 1 : 0;
        it.t += G;
        return true;
    }
    return false;
}

// Byte offset of B element (k, n) in the MN-major tile: column blocks of
// 128 bytes, each BK rows of 128 bytes with the same XOR swizzle.
template <int ES, int BK>
__device__ __forceinline__ uint32_t swz_mnmajor(int k, int n)
{
    constexpr int CW = 128 / ES;
    const int j = n / CW, nn = n - j * CW;
    const uint32_t nb = static_cast<uint32_t>(nn * ES);
    return static_cast<uint32_t>(j * BK * 128 + k * 128) +
           ((((nb >> 4) ^ static_cast<uint32_t>(k & 7)) << 4) | (nb & 15u));
}

// One A tensor map per residue class of row index (class-view A).
struct ClassMaps {
    CUtensorMap a[kMaxClasses];
};

// The GEMM of `args`, as a device routine: the part of the persistent tile
// schedule that falls to this CTA (CTAs blockIdx.x of gridDim.x, in pairs for
// CG == 2). Any kernel can call it once, with all of its threads, as one phase
// of a longer (persistent) kernel, provided that:
//   - the block has Traits::THREADS threads and at least Traits::SMEM_BYTES
//     of dynamic shared memory at smem_raw (the routine aligns it to 1024
//     bytes itself), and no other use of that shared memory overlaps the call;
//   - for CG == 2 the grid is launched in clusters of 2;
//   - every CTA of the grid calls it (the schedule spans the whole grid); for
//     stream-K layouts without a ticket counter (args.sk_ticket null) the
//     CTAs' slots follow blockIdx, so all of the grid must be resident at
//     once (with a ticket counter, slots follow the order the CTAs start in,
//     and no residency is assumed);
//   - tmA, tmB, tmC are tensor maps in parameter, constant or global memory,
//     encoded as the host entry points encode them (tmA points to one map,
//     or for class-view A to one map per residue class).
// On return the CTA's share of C is written; bulk stores are complete, and
// the CTA's tensor memory is freed. The routine's own work is all inside
// the call: nothing is left pending for the caller.
template <int DT, int BN, int CG, int PROD, int ST = 0>
__device__ __forceinline__ void gemm_cta(const CUtensorMap* tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                                         const GemmArgs& args, uint8_t* smem_raw)
{
    using T = Traits<DT, BN, CG, PROD, ST>;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Shared-memory carve-up (identical in both CTAs of a pair).
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + T::STAGES * T::A_BYTES;
    float* const epi = reinterpret_cast<float*>(gbase + T::STAGES * T::STAGE_BYTES);
    const uint32_t bars = base + T::STAGES * T::STAGE_BYTES + T::EPI_BYTES;
    uint8_t* const gbars = gbase + T::STAGES * T::STAGE_BYTES + T::EPI_BYTES;
    // barrier slots (8 bytes each)
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (T::STAGES + s); };
    auto tfull_bar = [&](int a) { return bars + 8u * (2 * T::STAGES + a); };
    auto tempty_bar = [&](int a) { return bars + 8u * (2 * T::STAGES + 2 + a); };
    const uint32_t drain_bar = bars + 8u * (2 * T::STAGES + 4);
    const uint32_t tmem_ready_bar = bars + 8u * (2 * T::STAGES + 5);   // pair: the peer's TMEM is allocated
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbars + 8 * (2 * T::STAGES + 6));
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbars + 8 * (2 * T::STAGES + 6) + 4);
    // C through the ring: per stage, a barrier for its C fill and a count of
    // the epilogue warps that have read their chunk of it.
    auto cfull_bar = [&](int s) { return bars + 8u * (2 * T::STAGES + 7 + s); };
    int* const c_readers = reinterpret_cast<int*>(gbars + 8 * (3 * T::STAGES + 7));
    // Stream-K: this launch's slot for the CTA (pair), from the ticket.
    volatile uint32_t* const slot_word =
        reinterpret_cast<volatile uint32_t*>(gbars + 8 * (3 * T::STAGES + 7) + 4 * T::STAGES);
    // Class-view A: per stage, the barrier a tile's first k-block of A lands
    // on when the fixer warp must zero its leading elements first.
    constexpr uint32_t kAfix = (8u * (3 * T::STAGES + 8) + 4u * T::STAGES + 7u) & ~7u;  // 8-byte aligned
    auto afix_bar = [&](int s) { return bars + kAfix + 8u * s; };
    static_assert(kAfix + 8 * T::STAGES <= T::BAR_BYTES, "barrier area");
    // Shared address of 4 KB slot j of ring stage s (its A part, then its B part).
    auto ring_slot = [&](int s, int j) -> uint32_t {
        constexpr int AS = T::A_BYTES / 4096;
        return j < AS ? sA + static_cast<uint32_t>(s * T::A_BYTES + j * 4096)
                      : sB + static_cast<uint32_t>(s * T::B_BYTES + (j - AS) * 4096);
    };
    // Class-view tiles hold rows P apart: their C goes out by rows, never as
    // bulk-store boxes.
    const int c_tma = T::CLS ? 0 : args.c_tma;
    // Class-view tiles whose C rows all share one 16-byte offset (c_cls).
    const bool c_cls = T::CLS && args.c_cls != 0;
    const bool c_ring = T::C_RING_OK && args.c_ring != 0 && c_tma != 0 && args.splits == 1 && args.sk_tiles == 0 &&
                        args.beta != 0.0f;

    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;

    // Stream-K slots are handed out in the order the CTAs (pairs) start: the
    // leader's first thread takes the next ticket. A final piece waits only on
    // slots before its own, whose CTAs have therefore started, so the fix-up
    // needs no co-residency: it finishes when other work holds SMs, or when
    // launches of this kind overlap on several streams (each with its own
    // counters). The atomic's latency overlaps the barrier set-up below.
    const bool ticketed = args.sk_tiles > 0 && args.sk_ticket != nullptr;
    unsigned ticket = 0;
    if (ticketed && leader && warp == 0 && lane == 0)
        ticket = atomicAdd(args.sk_ticket, 1u);

    // Barrier initialisation, spread over the lanes of warp 0: lane s < STAGES
    // takes ring stage s, the next two lanes the accumulator barriers, the
    // next one the rest.
    static_assert(T::STAGES + 3 <= 32, "one lane per stage");
    if (warp == 0) {
        if (lane < T::STAGES) {
            mbar_init(full_bar(lane), T::TMA ? 1 : T::NPW * 32);
            mbar_init(empty_bar(lane), 1);
            mbar_init(cfull_bar(lane), 1);
            if constexpr (T::CLS)
                mbar_init(afix_bar(lane), 1);
            c_readers[lane] = 0;
        } else if (lane < T::STAGES + 2) {
            mbar_init(tfull_bar(lane - T::STAGES), 1);
            mbar_init(tempty_bar(lane - T::STAGES), T::EPI_WARPS * CG);
        } else if (lane == T::STAGES + 2) {
            mbar_init(drain_bar, 1);
            mbar_init(tmem_ready_bar, 1);
            *abort_flag = 0;
        }
        fence_mbar_init();
    }
    if (T::TMA && warp == 0 && lane == 0) {
        for (int i = 0; i < (T::CLS ? args.a_classes : 1); ++i)
            tma_prefetch_desc(tmA + i);
        tma_prefetch_desc(&tmB);
    }
    if (c_tma && warp == T::EPI_WARP0 && lane == 0)
        tma_prefetch_desc(&tmC);
    if (ticketed && leader && warp == 0 && lane == 0) {
        // Launch sk_epoch takes tickets (sk_epoch - 1) * G .. sk_epoch * G - 1
        // (modulo 2^32): every CTA pair of every launch takes exactly one.
        const unsigned G = gridDim.x / CG;
        unsigned g = ticket - (args.sk_epoch - 1u) * G;
        if (g >= G) {   // cannot happen with one launch at a time per counter
            if (args.err)
                atomicOr(args.err, kErrTicket);
            g = blockIdx.x / CG;
        }
        *slot_word = g;
    }
    // Barrier initialisation is published to the CTA (and, for a pair, to
    // the peer); the producer then starts at once. Tensor memory is
    // allocated meanwhile and published only to the MMA and epilogue warps
    // (named barrier 1); in a pair the peer also tells the leader, whose MMAs
    // write the peer's tensor memory, through tmem_ready_bar.
    __syncthreads();
    if constexpr (CG == 2)
        cluster_sync();
    uint32_t tmem_base = 0;
    // The MMA warp and the epilogue warps (not the fixer warp of class-view
    // kernels): exactly the (1 + EPI_WARPS) warps named barrier 1 counts.
    if (warp >= T::MMA_WARP && warp < T::EPI_WARP0 + T::EPI_WARPS) {
        if (warp == T::MMA_WARP) {
            tmem_alloc<CG>(smem_u32(tmem_slot), T::TMEM_COLS);
            tmem_relinquish<CG>();
        }
        tc_fence_before();
        named_bar_sync(1, (1 + T::EPI_WARPS) * 32);
        tc_fence_after();
        tmem_base = *tmem_slot;
        if (CG == 2 && !leader && warp == T::MMA_WARP && lane == 0)
            mbar_arrive_cluster(map_to_cta(tmem_ready_bar, 0));
    }

    const WaitCtl wc{abort_flag, args.err, args.timeout_ns};
    // Barriers completed by TMA transactions or tcgen05.commit need only
    // CTA-scope acquire; the one barrier that the peer CTA's epilogue
    // arrives on with plain arrives (TMEM released) needs cluster scope.
    constexpr bool kClu = CG == 2;
    const int tile_step = gridDim.x / CG;
    // This CTA's slot: the ticket the leader took (published by the barriers
    // above: the CTA barrier, and for a pair the cluster barrier before the
    // peer reads the leader's word), else the launch order.
    int tile0 = blockIdx.x / CG;
    if (ticketed) {
        if constexpr (CG == 2)
            tile0 = leader ? static_cast<int>(*slot_word)
                           : static_cast<int>(ld_shared_cluster_u32(map_to_cta(smem_u32(
                                 const_cast<uint32_t*>(slot_word)), 0)));
        else
            tile0 = static_cast<int>(*slot_word);
    }

    if (warp < T::NPW) {
        // ------------------------------------------------------------ producer

        if constexpr (T::TMA) {
            if (lane == 0) {
                int stage = 0;
                uint32_t phase = 0;
                bool ok = true;
                // The pair's loads all complete on the leader's barrier.
                const uint32_t full0 = CG == 2 ? map_to_cta(full_bar(0), 0) : full_bar(0);
                WorkIter it = work_begin(args, tile0);
                Unit w;
                while (ok && work_next(args, tile_step, it, w)) {
                    // Class-view A: the tile's rows are view rows of class
                    // cls (rows cls + P*y), whose view starts ashift elements
                    // before each row; B follows that shift in K.
                    const int cls = T::CLS ? w.tm % args.a_classes : 0;
                    const int ashift = T::CLS ? args.a_shift[cls] : 0;
                    const int tmv = T::CLS ? w.tm / args.a_classes : w.tm;
                    const int m0 = tmv * (T::BM * CG) + static_cast<int>(rank) * T::BM;
                    const int n0 = w.tn * BN + static_cast<int>(rank) * T::BN_CTA;
                    for (int i = 0; i < w.kb1 - w.kb0; ++i) {
                        const int kb = w.rev ? w.kb1 - 1 - i : w.kb0 + i;
                        if (!wait_bar<false>(empty_bar(stage), phase ^ 1u, wc, kErrTimeoutProducer)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = full0 + 8u * stage;
                        const int k0 = kb * T::BK;
                        // The first operand (this CTA's 128 accumulator rows
                        // from m0) and the second (its BN_CTA columns from n0),
                        // each as it lies in memory: K-major as one box of
                        // BK x rows, MN-major as boxes of CW rows x BK. A
                        // swapped tile reads the first from B, the second from A.
                        const CUtensorMap* t1 = T::SWAP ? &tmB : tmA + cls;
                        const CUtensorMap* t2 = T::SWAP ? tmA : &tmB;
                        auto load = [&](uint32_t dst, const CUtensorMap* t, int x, int y) {
                            if constexpr (CG == 1)
                                tma_load_2d(dst, t, fb, x, y);
                            else
                                tma_load_2d_pair(dst, t, fb, x, y);
                        };
                        // In a pair only the leader arms the barrier, for both
                        // CTAs' bytes; the peer's copies just complete on it. A
                        // peer copy landing first drives the transaction count
                        // negative, which the barrier allows, and the leader's
                        // pending arrival keeps the phase open.
                        if (CG == 1 || leader)
                            mbar_arrive_expect_tx(full_bar(stage), CG * T::STAGE_BYTES);
                        if constexpr (T::A_MN) {
#pragma unroll
                            for (int j = 0; j < T::NBOX_A; ++j)
                                load(sA + stage * T::A_BYTES + j * (T::BK * 128), t1, m0 + j * T::CW, k0);
                        } else if constexpr (T::CLS) {
                            // A tile's first k-block reads ashift elements of the
                            // previous row in front of each row: it lands on this
                            // CTA's fix barrier, and the fixer warp zeroes them and
                            // completes the bytes on the full barrier.
                            if (kb == 0 && ashift > 0) {
                                mbar_arrive_expect_tx(afix_bar(stage), T::A_BYTES);
                                tma_load_2d(sA + stage * T::A_BYTES, t1, afix_bar(stage), k0, m0);
                            } else {
                                load(sA + stage * T::A_BYTES, t1, k0, m0);
                            }
                        } else {
                            load(sA + stage * T::A_BYTES, t1, k0, m0);
                        }
                        if constexpr (T::B_KM) {
                            load(sB + stage * T::B_BYTES, t2, k0, n0);
                        } else {
                            // Class-view A: K positions k0 - ashift .. of B (rows
                            // above 0 read as zero).
#pragma unroll
                            for (int j = 0; j < T::NBOX; ++j)
                                load(sB + stage * T::B_BYTES + j * (T::BK * 128), t2, n0 + j * T::CW, k0 - ashift);
                        }
                        if (++stage == T::STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    // Then this CTA's rows of the tile's C, column chunk by
                    // column chunk (the order the epilogue reads them in),
                    // each stage completing on this CTA's own cfull barrier.
                    if (ok && c_ring) {
                        const int crow = w.tm * (T::BM * CG) + static_cast<int>(rank) * T::BM;
                        const int ccol = w.tn * BN;
                        for (int cs = 0; cs < T::NCS; ++cs) {
                            if (!wait_bar<false>(empty_bar(stage), phase ^ 1u, wc, kErrTimeoutProducer)) {
                                ok = false;
                                break;
                            }
                            const int first = cs * T::CPS;
                            const int n = min(T::CPS, T::C_CHUNKS - first);
                            mbar_arrive_expect_tx(cfull_bar(stage), static_cast<uint32_t>(n) * 4096u);
                            for (int j = 0; j < n; ++j) {
                                const int id = first + j;
                                const int cc = id / (T::BM / 32), rb = id - cc * (T::BM / 32);
                                tma_load_2d(ring_slot(stage, j), &tmC, cfull_bar(stage), ccol + cc * 32, crow + rb * 32);
                            }
                            if (++stage == T::STAGES) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                    }
                }
                // Drain: wait until the MMA has released every stage filled
                // above, so no copy or commit is in flight when the CTA ends.
                if (ok) {
                    for (int i = 0; i < T::STAGES; ++i) {
                        if (!wait_bar<false>(empty_bar(stage), phase ^ 1u, wc, kErrTimeoutProducer))
                            break;
                        if (++stage == T::STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
        } else {
          // Row strides: dense plain-load kernels take them from K and N
          // themselves, measured 9-16% faster on the misaligned (8191, 4097,
          // 2049) shapes than reading separate strides; the strided kind
          // reads lda and ldb.
          const int sta = PROD == kProdPlain ? args.K : args.lda;
          const int stb = PROD == kProdPlain ? args.N : args.ldb;
          if constexpr (T::kTF32) {
            // Plain-load producer for 4-byte elements: asynchronous 4-byte
            // copies straight into the swizzled stage layout (A K-major,
            // B MN-major with 32-byte atoms: chunk c of row k at c ^ (k mod 4)),
            // zero-filled outside the matrix. Each thread commits one copy
            // group per fill and, STAGES - 1 fills later, waits for that
            // group, makes it visible to the tensor core (proxy fence) and
            // arrives on the fill's barrier.
            const uint32_t* __restrict__ gA = static_cast<const uint32_t*>(args.A);
            const uint32_t* __restrict__ gB = static_cast<const uint32_t*>(args.B);
            constexpr int NP = T::NPW * 32;
            static_assert(NP == 128 && T::BK == 32 && BN % NP == 0, "copy layout: 128 threads, 32-wide K");
            constexpr int LAG = T::STAGES - 1;
            constexpr int BCOLS = BN / NP;     // B columns per thread: n = p + 128 c
            const int p = threadIdx.x;         // producer warps are warps 0..NPW-1
            const int ak = p & 31;             // this thread's k within every A row
            const int ar0 = p >> 5;            // its first A row; rows ar0 + 4 i
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int fills = 0, signalled = 0;
            WorkIter it = work_begin(args, tile0);
            Unit w;
            while (ok && work_next(args, tile_step, it, w)) {
                const int m0 = w.tm * T::BM;
                const int n0 = w.tn * BN;
                for (int i = 0; i < w.kb1 - w.kb0; ++i) {
                    const int kb = w.rev ? w.kb1 - 1 - i : w.kb0 + i;
                    if (!wait_bar<false>(empty_bar(stage), phase ^ 1u, wc, kErrTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    const int k0 = kb * T::BK;
                    const uint32_t dA = sA + stage * T::A_BYTES;
                    const uint32_t dB = sB + stage * T::B_BYTES;
                    const int gk = k0 + ak;
#pragma unroll 8
                    for (int i = 0; i < T::BM / 4; ++i) {
                        const int r = ar0 + 4 * i;
                        const int gr = m0 + r;
                        const bool v = gk < args.K && gr < args.M;
                        const uint32_t* src = v ? gA + static_cast<int64_t>(gr) * sta + gk : gA;
                        cp_async_4(dA + static_cast<uint32_t>(r * 128 + ((((ak >> 2) ^ (r & 7)) << 4) | ((ak & 3) << 2))),
                                   src, v ? 4u : 0u);
                    }
#pragma unroll
                    for (int c = 0; c < BCOLS; ++c) {
                        const int n = p + NP * c;
                        const int gn = n0 + n;
                        const int nn = n & 31;
                        const uint32_t col = dB + static_cast<uint32_t>((n >> 5) * (T::BK * 128) + ((nn & 7) << 2));
#pragma unroll 8
                        for (int kr = 0; kr < T::BK; ++kr) {
                            const int gk2 = k0 + kr;
                            const bool v = gn < args.N && gk2 < args.K;
                            const uint32_t* src = v ? gB + static_cast<int64_t>(gk2) * stb + gn : gB;
                            cp_async_4(col + static_cast<uint32_t>(kr * 128 + ((((nn >> 3) ^ (kr & 3)) << 5))), src,
                                       v ? 4u : 0u);
                        }
                    }
                    cp_async_commit();
                    ++fills;
                    if (fills - signalled > LAG) {
                        cp_async_wait<LAG>();
                        fence_proxy_async_smem();
                        mbar_arrive(full_bar(signalled % T::STAGES));
                        ++signalled;
                    }
                    if (++stage == T::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Every copy lands before the CTA moves on; signal the fills still open.
            cp_async_wait<0>();
            fence_proxy_async_smem();
            for (; signalled < fills; ++signalled)
                mbar_arrive(full_bar(signalled % T::STAGES));
            if (ok) {
                for (int i = 0; i < T::STAGES; ++i) {
                    if (!wait_bar<false>(empty_bar(stage), phase ^ 1u, wc, kErrTimeoutProducer))
                        break;
                    if (++stage == T::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
          } else {
            // Plain-load producer (1-SM, 2-byte elements): any row stride.
            using E = uint16_t;
            const E* __restrict__ gA = static_cast<const E*>(args.A);
            const E* __restrict__ gB = static_cast<const E*>(args.B);
            constexpr int NP = T::NPW * 32;
            constexpr int BATCH = 16;
            const int p = threadIdx.x;  // producer warps are warps 0..NPW-1
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            WorkIter it = work_begin(args, tile0);
            Unit w;
            while (ok && work_next(args, tile_step, it, w)) {
                const int m0 = w.tm * T::BM;
                const int n0 = w.tn * BN;
                for (int i = 0; i < w.kb1 - w.kb0; ++i) {
                    const int kb = w.rev ? w.kb1 - 1 - i : w.kb0 + i;
                    if (!wait_bar<false>(empty_bar(stage), phase ^ 1u, wc, kErrTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    const int k0 = kb * T::BK;
                    uint8_t* const dA = gbase + (sA - base) + stage * T::A_BYTES;
                    uint8_t* const dB = gbase + (sB - base) + stage * T::B_BYTES;
                    // A tile: BM x BK, consecutive threads take consecutive k.
                    constexpr int NA = T::BM * T::BK / NP;
                    static_assert(NA % BATCH == 0, "A batch");
#pragma unroll 1
                    for (int i0 = 0; i0 < NA; i0 += BATCH) {
                        E v[BATCH];
#pragma unroll
                        for (int i = 0; i < BATCH; ++i) {
                            const int idx = p + (i0 + i) * NP;
                            const int r = idx / T::BK, k = idx - r * T::BK;
                            const int gm = m0 + r, gk = k0 + k;
                            v[i] = (gm < args.M && gk < args.K) ? __ldg(gA + static_cast<int64_t>(gm) * sta + gk)
                                                                : E(0);
                        }
#pragma unroll
                        for (int i = 0; i < BATCH; ++i) {
                            const int idx = p + (i0 + i) * NP;
                            const int r = idx / T::BK, k = idx - r * T::BK;
                            *reinterpret_cast<E*>(dA + swz_kmajor<T::ES>(r, k)) = v[i];
                        }
                    }
                    // B tile: BK x BN, consecutive threads take consecutive n.
                    constexpr int NB = T::BK * BN / NP;
                    static_assert(NB % BATCH == 0, "B batch");
#pragma unroll 1
                    for (int i0 = 0; i0 < NB; i0 += BATCH) {
                        E v[BATCH];
#pragma unroll
                        for (int i = 0; i < BATCH; ++i) {
                            const int idx = p + (i0 + i) * NP;
                            const int kr = idx / BN, n = idx - kr * BN;
                            const int gk = k0 + kr, gn = n0 + n;
                            v[i] = (gk < args.K && gn < args.N) ? __ldg(gB + static_cast<int64_t>(gk) * stb + gn)
                                                                : E(0);
                        }
#pragma unroll
                        for (int i = 0; i < BATCH; ++i) {
                            const int idx = p + (i0 + i) * NP;
                            const int kr = idx / BN, n = idx - kr * BN;
                            *reinterpret_cast<E*>(dB + swz_mnmajor<T::ES, T::BK>(kr, n)) = v[i];
                        }
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(full_bar(stage));
                    if (++stage == T::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (ok) {
                for (int i = 0; i < T::STAGES; ++i) {
                    if (!wait_bar<false>(empty_bar(stage), phase ^ 1u, wc, kErrTimeoutProducer))
                        break;
                    if (++stage == T::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
          }
        }
    } else if (warp == T::MMA_WARP) {
        // ----------------------------------------------------------------- MMA
        if (leader && lane == 0) {
            int stage = 0;
            uint32_t fpar = 0;  // per stage: parity of its next k-block fill (C fills skip the full barrier)
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true, issued = false;
            if constexpr (CG == 2)
                ok = wait_bar<true>(tmem_ready_bar, 0, wc, kErrTimeoutMma);
            WorkIter it = work_begin(args, tile0);
            Unit w;
            while (ok && work_next(args, tile_step, it, w)) {
                // The peer's epilogue releases the accumulator too: cluster scope.
                if (!wait_bar<kClu>(tempty_bar(acc), acc_phase ^ 1u, wc, kErrTimeoutMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * T::ACC_COLS);
                // Class-view A in a pair: a tile's first k-block may be completed
                // by the peer's fixer (plain stores, then a cluster-scope fence
                // and complete_tx), so that wait acquires at cluster scope.
                const bool fix0 = T::CLS && CG == 2 && w.kb0 == 0 && args.a_shift[w.tm % args.a_classes] > 0;
                for (int i = 0; i < w.kb1 - w.kb0; ++i) {
                    const int kb = w.rev ? w.kb1 - 1 - i : w.kb0 + i;
                    const bool got = fix0 && kb == 0
                                         ? wait_bar<kClu>(full_bar(stage), (fpar >> stage) & 1u, wc, kErrTimeoutMma)
                                         : wait_bar<false>(full_bar(stage), (fpar >> stage) & 1u, wc, kErrTimeoutMma);
                    if (!got) {
                        ok = false;
                        break;
                    }
                    fpar ^= 1u << stage;
                    tc_fence_after();
                    const uint32_t a0 = sA + stage * T::A_BYTES;
                    const uint32_t b0 = sB + stage * T::B_BYTES;
#pragma unroll
                    for (int ks = 0; ks < T::KSTEPS; ++ks) {
                        // K-major operands: 128-byte rows, one MMA step of K
                        // 32 bytes on; MN-major: column blocks BK*128 bytes
                        // apart, one MMA step of K UK rows on.
                        const uint64_t ad = T::A_MN ? sdesc(a0 + ks * T::MN_KSTEP, T::MN_LBO, T::MN_SBO, T::MN_LAYOUT)
                                                    : sdesc(a0 + ks * T::K_KSTEP, 16, 1024, kLayoutSW128);
                        const uint64_t bd = T::B_KM ? sdesc(b0 + ks * T::K_KSTEP, 16, 1024, kLayoutSW128)
                                                    : sdesc(b0 + ks * T::MN_KSTEP, T::MN_LBO, T::MN_SBO, T::MN_LAYOUT);
                        mma_ss<CG, T::kTF32>(d, ad, bd, T::IDESC, (i != 0 || ks != 0) ? 1u : 0u);
                    }
                    issued = true;
                    if constexpr (CG == 1)
                        mma_commit(empty_bar(stage));
                    else
                        mma_commit_pair(empty_bar(stage), 0x3);
                    if (++stage == T::STAGES)
                        stage = 0;
                }
                if (!ok)
                    break;
                if constexpr (CG == 1)
                    mma_commit(tfull_bar(acc));
                else
                    mma_commit_pair(tfull_bar(acc), 0x3);
                if (c_ring) {  // the tile's C stages go to the epilogue
                    stage += T::NCS;
                    if (stage >= T::STAGES)
                        stage -= T::STAGES;
                }
                acc ^= 1;
                if (acc == 0)
                    acc_phase ^= 1u;
            }
            if (!ok && issued) {
                // Let issued MMAs finish before tensor memory is freed.
                if constexpr (CG == 1)
                    mma_commit(drain_bar);
                else
                    mma_commit_pair(drain_bar, 0x1);
                const WaitCtl dw{abort_flag, args.err, args.timeout_ns};
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait<kClu>(drain_bar, 0)) {
                    if (globaltimer_ns() - t0 > dw.timeout_ns) {
                        if (args.err)
                            atomicOr(args.err, kErrTimeoutDrain);
                        break;
                    }
                }
            }
        }
    } else if (T::CLS && warp == T::FIX_WARP) {
        // --------------------------------------------------------------- fixer
        // Class-view A: a tile's first k-block reads, in front of each row, the
        // ashift elements of memory that precede it (the view starts aligned
        // down). Once that block has landed, zero those elements of all 128
        // rows (K-major, 128-byte swizzle), make the stores visible to the
        // tensor core and complete the block's bytes on the full barrier (the
        // pair leader's), which the producer left open for them.
        if constexpr (T::CLS) {
            int stage = 0;
            uint32_t apar = 0;  // per stage: parity of its next fix
            const uint32_t full0 = CG == 2 ? map_to_cta(full_bar(0), 0) : full_bar(0);
            WorkIter it = work_begin(args, tile0);
            Unit w;
            while (work_next(args, tile_step, it, w)) {
                const int ashift = args.a_shift[w.tm % args.a_classes];
                if (w.kb0 == 0 && ashift > 0) {
                    // k-block 0 is the unit's first stage, or its last when the
                    // unit runs through K backwards.
                    const int fs = w.rev ? (stage + (w.kb1 - w.kb0 - 1)) % T::STAGES : stage;
                    if (!wait_bar<false>(afix_bar(fs), (apar >> fs) & 1u, wc, kErrTimeoutProducer))
                        break;
                    apar ^= 1u << fs;
                    const uint32_t a0 = sA + fs * T::A_BYTES;
                    for (int i = lane; i < T::BM * ashift; i += 32) {
                        const int row = i / ashift, k = i - row * ashift;
                        if constexpr (T::ES == 4)
                            st_shared_u32(a0 + swz_kmajor<4>(row, k), 0u);
                        else
                            st_shared_u16(a0 + swz_kmajor<2>(row, k), static_cast<uint16_t>(0));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        fence_acq_rel_cluster();
                        mbar_complete_tx_cluster(full0 + 8u * fs, T::A_BYTES);
                    }
                    __syncwarp();
                }
                stage = (stage + (w.kb1 - w.kb0)) % T::STAGES;
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - T::EPI_WARP0;      // 0..7
        const int sub = warp & 3;                // TMEM lane quarter this warp may access
        constexpr int CSTEP = T::EPI_WARPS / 4;  // warps per TMEM lane quarter
        const int half = ew >> 2;                // this warp takes chunks half, half + CSTEP, ...
        float* const buf = epi + ew * (T::EPI_WARP_BYTES / 4);
        const uint32_t sb = smem_u32(buf);       // 1024-byte aligned
        const uint32_t tempty0 = CG == 2 ? map_to_cta(tempty_bar(0), 0) : tempty_bar(0);
        int acc = 0;
        uint32_t acc_phase = 0;
        const float alpha = args.alpha, beta = args.beta;
        const int ldc = args.ldc;
        constexpr int NCHUNK = BN / 32;
        // C's element address (fp32): row r starts (c_el + r * ldc) mod 4
        // elements past a 16-byte boundary.
        const uint64_t c_el = reinterpret_cast<uintptr_t>(args.C) >> 2;
        // C values (bulk-store path, beta != 0) of row (row0 + lane), columns
        // gcol0 .. gcol0 + 31, as 8 aligned float4 loads; zero outside M x N.
        auto load_c = [&](float (&cv)[32], int grow, int gcol0) {
            const float4* src = reinterpret_cast<const float4*>(args.C + static_cast<int64_t>(grow) * ldc + gcol0);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (grow < args.M && gcol0 + 4 * q < args.N)
                    x = src[q];
                cv[4 * q] = x.x;
                cv[4 * q + 1] = x.y;
                cv[4 * q + 2] = x.z;
                cv[4 * q + 3] = x.w;
            }
        };
        // The tile loop, compiled twice: with C through the ring, and with C
        // loaded by the epilogue (or not read), so that each copy keeps only
        // the registers its own path needs.
        WorkIter it = work_begin(args, tile0);
        bool ok = true;
        auto tile_loop = [&](auto mode_tag) {
            constexpr int MODE = decltype(mode_tag)::value;
            constexpr bool RING = MODE == 1;  // C through the operand ring
            constexpr bool SK = MODE == 2;    // stream-K pieces
            // beta != 0 (only unsplit): the plain copy reads each chunk's C
            // ahead (the first one before the accumulator wait); the
            // stream-K copy reads it only when the chunk is stored, after any
            // partial sums have been added, to keep its registers in bounds.
            const bool prefetch_c = MODE == 0 && !T::SWAP && c_tma && beta != 0.0f;
            const bool late_c = SK && !T::SWAP && c_tma && beta != 0.0f;
            // Row-store path (C not 16-byte aligned), beta != 0: each chunk's
            // 32 rows of C at this lane's column are loaded together, all in
            // flight at once, the first chunk's before the accumulator wait.
            const bool rows_c = MODE == 0 && !T::SWAP && !c_tma && beta != 0.0f;
            // C through the ring: where the next unit's stages start, and per
            // stage the parity of its next C fill.
            int rpos = 0;
            uint32_t cpar = 0;
            Unit w;
            // The stream-K copy takes this CTA's stream-K pieces; the others
            // take whole units (all of them, or those after the pieces).
            while (ok && (SK ? it.pos < it.end : true) && work_next<SK>(args, tile_step, it, w)) {
                // Class-view tiles: view rows of class cls, actual rows
                // cls + P * (view row).
                const int ncls = T::CLS ? args.a_classes : 1;
                const int cls = T::CLS ? w.tm % ncls : 0;
                const int row0 = (T::CLS ? w.tm / ncls : w.tm) * (T::BM * CG) + static_cast<int>(rank) * T::BM + sub * 32;
                const int n0 = w.tn * BN;
                // Row-store addressing of this warp's 32 rows: the first one's
                // element offset (before the column), the step between rows
                // and how many lie inside C. Split s writes its slice of the
                // output: rows s * out_rows + row.
                const int yoff = w.s * args.out_rows;
                int cst = 0;  // ring stage holding this tile's first C chunks
                if constexpr (RING) {
                    cst = (rpos + (w.kb1 - w.kb0)) % T::STAGES;
                    rpos = (cst + T::NCS) % T::STAGES;
                }
                // Read the first chunk's C before waiting for the accumulator, so
                // its latency overlaps the main loop; later chunks read theirs in turn.
                float cv[32];
                if constexpr (!RING) {
                    if (prefetch_c) {
                        load_c(cv, row0 + lane, n0 + half * 32);
                    } else if (rows_c) {
                        // Row-store path: the first chunk's 32 rows at this
                        // lane's column, loaded before the accumulator wait too.
                        const int col = n0 + half * 32 + lane;
                        const int64_t rb =
                            (static_cast<int64_t>(yoff) + (T::CLS ? cls + ncls * row0 : row0)) * ldc + col;
                        const int64_t rs = T::CLS ? static_cast<int64_t>(ncls) * ldc : static_cast<int64_t>(ldc);
                        const int nr = T::CLS ? min(32, args.a_rows[cls] - row0) : min(32, args.M - row0);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            cv[i] = i < nr && col < args.N ? c_load(args.C, args.c_half, rb + i * rs) : 0.0f;
                    }
                }
                if (!wait_bar<false>(tfull_bar(acc), acc_phase, wc, kErrTimeoutEpilogue))
                    break;
                tc_fence_after();
                if constexpr (SK) {
                    // Stream-K final piece: the partial tiles of slots
                    // w.first .. tile0 - 1 (same rows of the same tile) must
                    // have been written before they are added below.
                    if (w.kind == kSkFinal) {
                        if (lane == 0) {
                            for (int j = w.first; ok && j < tile0; ++j)
                                ok = wait_counter(args.sk_flags + j * CG + static_cast<int>(rank),
                                                  args.sk_epoch * static_cast<unsigned>(T::EPI_WARPS), wc,
                                                  kErrTimeoutPartial);
                        }
                        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                        if (!ok)
                            break;
                    }
                }
                const uint32_t tbase = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) +
                                       static_cast<uint32_t>(acc * T::ACC_COLS);
                if constexpr (NCHUNK < CSTEP) {
                    // A tile narrower than the epilogue's warps: a warp with
                    // no chunk still hands the accumulator back.
                    if (half >= NCHUNK) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if constexpr (CG == 1)
                                mbar_arrive(tempty0 + 8u * acc);
                            else
                                mbar_arrive_cluster(tempty0 + 8u * acc);
                        }
                    }
                }
#pragma unroll 1
                for (int c = half; c < NCHUNK; c += CSTEP) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, r);
                    tmem_wait_ld();
                    if (c + CSTEP >= NCHUNK) {
                        // This warp's TMEM reads of the accumulator are done: hand it back.
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if constexpr (CG == 1)
                                mbar_arrive(tempty0 + 8u * acc);
                            else
                                mbar_arrive_cluster(tempty0 + 8u * acc);
                        }
                    }
                    const int gcol0 = n0 + c * 32;
                    if constexpr (SK) {
                        // Partial tile of slot g, as [column chunk][16-byte
                        // piece q][row]: lane-consecutive 16-byte pieces, so
                        // both the writer and the reader move whole lines.
                        if (w.kind != kWhole) {
                            const int row = sub * 32 + lane;
                            if (w.kind == kSkPartial) {
                                float* slot =
                                    args.sk_ws + static_cast<int64_t>(tile0 * CG + static_cast<int>(rank)) * (128 * BN);
#pragma unroll
                                for (int q = 0; q < 8; ++q)
                                    st_global_v4(slot + ((c * 8 + q) * 128 + row) * 4, __uint_as_float(r[4 * q]),
                                                 __uint_as_float(r[4 * q + 1]), __uint_as_float(r[4 * q + 2]),
                                                 __uint_as_float(r[4 * q + 3]));
                                continue;
                            }
                            // Final piece: add the earlier slots' partial sums,
                            // in ascending slot order.
#pragma unroll 1
                            for (int j = w.first; j < tile0; ++j) {
                                const float* slot =
                                    args.sk_ws + static_cast<int64_t>(j * CG + static_cast<int>(rank)) * (128 * BN);
#pragma unroll
                                for (int q = 0; q < 8; ++q) {
                                    float p[4];
                                    ld_global_cg_v4(slot + ((c * 8 + q) * 128 + row) * 4, p[0], p[1], p[2], p[3]);
#pragma unroll
                                    for (int e = 0; e < 4; ++e)
                                        r[4 * q + e] = __float_as_uint(__uint_as_float(r[4 * q + e]) + p[e]);
                                }
                            }
                        }
                    }
                    if constexpr (T::SWAP) {
                        // Swapped tile: this lane's accumulator row is column
                        // ccol of C, and its 32 values are rows crow .. crow + 31.
                        // For each row j the warp touches 32 consecutive floats.
                        const int ccol = row0 + lane;
                        const int crow = gcol0;
                        float ct[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            ct[j] = beta != 0.0f && crow + j < args.M && ccol < args.N
                                        ? c_load(args.C, args.c_half, static_cast<int64_t>(crow + j) * ldc + ccol)
                                        : 0.0f;
                        if (c_tma) {
                            // Stage the 32 x 32 block of C (rows crow.., columns
                            // row0..) in the store's 128-byte swizzle: row j, piece
                            // lane / 4 at (lane / 4) ^ (j & 7); conflict free.
                            if (lane == 0)
                                bulk_wait_read<0>();
                            __syncwarp();
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                float v = alpha * __uint_as_float(r[j]);
                                if (beta != 0.0f)
                                    v = fmaf(beta, ct[j], v);
                                st_shared_f32(sb + static_cast<uint32_t>(j * 128 + ((((lane >> 2) ^ (j & 7)) << 4) |
                                                                                    ((lane & 3) << 2))),
                                              v);
                            }
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0 && crow < args.M && row0 < args.N) {
                                tma_store_2d(&tmC, sb, row0, yoff + crow);
                                bulk_commit();
                            }
                        } else if (ccol < args.N) {
                            const int64_t c0 = (static_cast<int64_t>(yoff) + crow) * ldc + ccol;
                            const int rows = min(32, args.M - crow);
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                if (j < rows) {
                                    float v = alpha * __uint_as_float(r[j]);
                                    if (beta != 0.0f)
                                        v = fmaf(beta, ct[j], v);
                                    c_store(args.C, args.c_half, c0 + static_cast<int64_t>(j) * ldc, v);
                                }
                            }
                        }
                        continue;
                    }
                    if (c_tma) {
                        // Bulk-store path: this thread owns row (row0 + lane) of the
                        // 32 x 32 chunk. Stage it in the store's 128-byte swizzle
                        // (16-byte piece q of row l at position q ^ (l & 7): each
                        // group of 8 lanes covers all 32 banks) and let one lane
                        // hand the chunk to the TMA engine, which clips it to M x N.
                        const int grow = row0 + lane;
                        // C through the ring: chunk (column chunk c, row block sub)
                        // of the tile's C, in the same swizzle, in slot csrc of
                        // stage cst_c once its fill has landed.
                        int cs = 0, cst_c = 0;
                        uint32_t csrc = 0;
                        if constexpr (RING) {
                            const int id = c * (T::BM / 32) + sub;
                            cs = id / T::CPS;
                            cst_c = cst + cs < T::STAGES ? cst + cs : cst + cs - T::STAGES;
                            if (!wait_bar<false>(cfull_bar(cst_c), (cpar >> cst_c) & 1u, wc, kErrTimeoutEpilogue)) {
                                ok = false;
                                break;
                            }
                            csrc = ring_slot(cst_c, id - cs * T::CPS) + static_cast<uint32_t>(lane * 128);
                        } else if ((prefetch_c && c != half) || late_c) {
                            load_c(cv, grow, gcol0);
                        }
                        if (lane == 0)
                            bulk_wait_read<0>();  // the previous store has finished reading the buffer
                        __syncwarp();
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const uint32_t piece = static_cast<uint32_t>((q ^ (lane & 7)) << 4);
                            float v[4], cq[4];
                            if constexpr (RING) {
                                ld_shared_v4(csrc + piece, cq[0], cq[1], cq[2], cq[3]);
                            } else {
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    cq[e] = cv[4 * q + e];
                            }
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                v[e] = alpha * __uint_as_float(r[4 * q + e]);
                                if (beta != 0.0f)
                                    v[e] = fmaf(beta, cq[e], v[e]);
                            }
                            st_shared_v4(sb + static_cast<uint32_t>(lane * 128) + piece, v[0], v[1], v[2], v[3]);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (row0 < args.M && gcol0 < args.N) {
                                tma_store_2d(&tmC, sb, gcol0, yoff + row0);
                                bulk_commit();
                            }
                            // This warp has read its chunk of the C stage; the
                            // stage's last reader hands it back to the producer.
                            if constexpr (RING) {
                                const int readers = min(T::CPS, T::C_CHUNKS - cs * T::CPS);
                                __threadfence_block();
                                if (atomicAdd(&c_readers[cst_c], 1) == readers - 1) {
                                    atomicSub(&c_readers[cst_c], readers);
                                    __threadfence_block();
                                    mbar_arrive(empty_bar(cst_c));
                                }
                            }
                        }
                        continue;
                    }
                    // Row-store fallback: transpose through the XOR-swizzled
                    // buffer (element (row l, column j) at l*32 + (j ^ l): conflict
                    // free both ways), then each row is written by the warp as 32
                    // consecutive floats, masked to M x N.
                    const int col = gcol0 + lane;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        buf[lane * 32 + (j ^ lane)] = __uint_as_float(r[j]);
                    // This warp's 32 rows: the first one's element offset at
                    // this column, the step between rows, how many lie in C.
                    // Split s writes its slice of the output (rows s * out_rows
                    // + row); class-view rows are cls + P * (view row).
                    const int64_t c0 =
                        (static_cast<int64_t>(yoff) + (T::CLS ? cls + ncls * row0 : row0)) * ldc + col;
                    const int64_t rstep = T::CLS ? static_cast<int64_t>(ncls) * ldc : static_cast<int64_t>(ldc);
                    const int nrows = T::CLS ? min(32, args.a_rows[cls] - row0) : min(32, args.M - row0);
                    // beta != 0: the chunk's C at this column, all 32 loads in
                    // flight at once (the accumulator values now sit in the
                    // buffer, which frees their registers).
                    if constexpr (!RING) {
                        if (rows_c && c != half) {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                cv[i] = i < nrows && col < args.N ? c_load(args.C, args.c_half, c0 + i * rstep) : 0.0f;
                        }
                    }
                    __syncwarp();
                    // This class's rows start s elements past a 16-byte boundary.
                    const int s = T::CLS ? static_cast<int>((c_el + static_cast<uint64_t>(cls + ncls * row0) * ldc) & 3u)
                                         : 0;
                    if constexpr (T::CLS && MODE == 0) {
                        if (c_cls && gcol0 + 32 <= args.N && (s == 0 || args.c_cls == 2)) {
                            // Class-view tiles, fp32 C whose rows P apart lie a
                            // whole number of 16-byte units apart: every row of
                            // the chunk starts s elements past a 16-byte boundary.
                            // Columns lo .. lo + w - 1 of each row (lo = (4 - s) %
                            // 4, w = 32 or 28) leave in 16-byte stores, lanes on
                            // consecutive 16-byte units; the other 4 - s + s
                            // columns (at the chunk's two ends, in 16-byte units
                            // shared with the neighbouring chunks) go element by
                            // element, one row per lane. A chunk that reaches
                            // past column N, and (c_cls == 1) misaligned rows,
                            // take the row stores below.
                            float v[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                v[i] = alpha * buf[i * 32 + (lane ^ i)];
                                if (beta != 0.0f)
                                    v[i] = fmaf(beta, cv[i], v[i]);
                            }
                            __syncwarp();
                            const int lo = s ? 4 - s : 0, w = s ? 28 : 32;
                            // Stage: columns lo .. lo + w - 1 as rows of w floats,
                            // then the 4 edge columns (the first lo, the last s).
                            const int bc = lane - lo;
                            if (bc >= 0 && bc < w) {
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    buf[i * w + bc] = v[i];
                            } else {
                                const int e = lane < lo ? lane : lane - w;
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    buf[32 * 28 + i * 4 + e] = v[i];
                            }
                            __syncwarp();
                            // 16-byte unit u = t * 32 + lane of the w / 4 per row.
#pragma unroll
                            for (int t = 0; t < 8; ++t) {
                                const int u = t * 32 + lane;
                                const int row = s ? u / 7 : u >> 3;
                                const int g = u - row * (w >> 2);
                                if (row < min(nrows, 32)) {
                                    float x0, x1, x2, x3;
                                    ld_shared_v4(sb + static_cast<uint32_t>(u * 16), x0, x1, x2, x3);
                                    st_global_v4(args.C + static_cast<int64_t>(cls + ncls * (row0 + row)) * ldc + gcol0 + lo +
                                                     4 * g,
                                                 x0, x1, x2, x3);
                                }
                            }
                            if (s != 0 && lane < nrows) {
                                const int64_t e0 = static_cast<int64_t>(cls + ncls * (row0 + lane)) * ldc + gcol0;
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    args.C[e0 + (e < lo ? e : e + 28)] = buf[32 * 28 + lane * 4 + e];
                            }
                            __syncwarp();
                            continue;
                        }
                    }
                    if (col < args.N) {
                        const int kind = args.c_half;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            if (i < nrows) {
                                float v = alpha * buf[i * 32 + (lane ^ i)];
                                if (beta != 0.0f)
                                    v = fmaf(beta, rows_c ? cv[i] : c_load(args.C, kind, c0 + i * rstep), v);
                                c_store(args.C, kind, c0 + i * rstep, v);
                            }
                        }
                    }
                    __syncwarp();
                }
                if constexpr (RING) {
                    for (int cs = 0; cs < T::NCS; ++cs)
                        cpar ^= 1u << (cst + cs < T::STAGES ? cst + cs : cst + cs - T::STAGES);
                } else if constexpr (SK) {
                    if (w.kind == kSkPartial) {
                        // Publish this warp's share of the partial tile.
                        __threadfence();
                        __syncwarp();
                        if (lane == 0)
                            red_release_add(args.sk_flags + tile0 * CG + static_cast<int>(rank), 1u);
                    }
                }
                acc ^= 1;
                if (acc == 0)
                    acc_phase ^= 1u;
            }
        };
        using Plain = std::integral_constant<int, 0>;
        using Ring = std::integral_constant<int, 1>;
        using StreamK = std::integral_constant<int, 2>;
        if (T::TMA && args.sk_tiles > 0) {
            // Stream-K pieces first, then the whole tiles in the plain copy
            // (the pieces' extra work does not weigh on its registers).
            if constexpr (T::TMA)
                tile_loop(StreamK{});
            tile_loop(Plain{});
        } else if (T::C_RING_OK && c_ring) {
            if constexpr (T::C_RING_OK)
                tile_loop(Ring{});
        } else {
            tile_loop(Plain{});
        }
        if (c_tma && lane == 0) {
            bulk_wait<0>();  // every bulk store of this warp has completed
            fence_proxy_async_global();
        }
        __syncwarp();
    }

    // ------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2)
        cluster_sync();
    if (warp == T::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, T::TMEM_COLS);
    }
}

template <int DT, int BN, int CG, int PROD, int ST>
__global__ void __launch_bounds__(Traits<DT, BN, CG, PROD, ST>::THREADS, 1)
    sat_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const GemmArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    gemm_cta<DT, BN, CG, PROD, ST>(&tmA, tmB, tmC, args, smem_raw);
}

template <int DT, int BN, int CG, int ST>
__global__ void __launch_bounds__(Traits<DT, BN, CG, kProdClassA, ST>::THREADS, 1)
    sat_gemm_cls_kernel(const __grid_constant__ ClassMaps tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const GemmArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    gemm_cta<DT, BN, CG, kProdClassA, ST>(tmA.a, tmB, tmC, args, smem_raw);
}

}  // namespace sat
