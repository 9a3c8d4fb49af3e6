// Shape-adaptive choice of tile and schedule.
//
// "Measured data point on fixed-tile vs shape-adaptive GEMM" (section "The
// wall, and why we think it's structural", and section 2.1 of the matching
// post-mortem "Post-mortem: a GPU stack without nvcc, cuBLAS, or LLVM")
// reports that one fixed 128x128 tile reaches parity in one band of shapes
// and loses outside it, and that the schedule, not only the tile size, was
// the binding term. The FlashInfer pull request "fix(fp4_gemm autotune) SM107
// kernel family excluded from autotune candidates" adds that the tile count
// against the SM count (wave quantization) and the raster order both swing
// throughput. So the choice here covers tile N, CTA pair vs single SM,
// raster order and raster group, in two steps:
//   1. an exact (dtype, M, N, K) hit in the committed sweep table
//      (sweep_table.inc, written from on-device measurements), else
//   2. a power-of-two bucket hit: the table row whose M, N and K round up to
//      the same powers of two (the nearest such row, same load path), as
//      FlashInfer's autotuner keys its lazily filled buckets, else
//   3. an analytic rule: estimated time = waves x per-tile time, where
//      waves = ceil(tiles / concurrent tiles) and a tile costs the larger of
//      its tensor-core time and its operand-fill time; the raster order and
//      group are those with the least estimated operand traffic from DRAM
//      (operand_traffic, below).
#include "dispatch.h"

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <utility>
#include <vector>

namespace sat {

namespace {

struct TableRow {
    int dt;
    int64_t M, N, K;
    Choice c;
};

const TableRow kTable[] = {
#include "sweep_table.inc"
};

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Effective L2 capacity for operand panels (of 129 MB), see select_config.
constexpr double kL2Effective = 60e6;

// ceil(log2(x)) for x >= 1.
int log2_ceil(int64_t x)
{
    int b = 0;
    while ((int64_t(1) << b) < x)
        ++b;
    return b;
}

// Whether TMA can read the operands of a dense row-major problem.
bool tma_rows(int64_t K, int64_t N, int dt)
{
    const int64_t es = dt == 0 ? 4 : 2;
    return (K * es) % 16 == 0 && (N * es) % 16 == 0;
}

// Output tile (tm, tn) of tile index t in raster order (as the kernel maps it).
void coord(int64_t t, int64_t tiles_m, int64_t tiles_n, int raster, int group, int64_t* tm, int64_t* tn)
{
    if (raster == 0) {
        const int64_t per = group * tiles_n, g = t / per, r = t - g * per, first = g * group;
        const int64_t gs = std::min<int64_t>(group, tiles_m - first);
        *tm = first + r % gs;
        *tn = r / gs;
    } else {
        const int64_t per = group * tiles_m, g = t / per, r = t - g * per, first = g * group;
        const int64_t gs = std::min<int64_t>(group, tiles_n - first);
        *tn = first + r % gs;
        *tm = r / gs;
    }
}

}  // namespace

double operand_traffic(int64_t tiles_m, int64_t tiles_n, int64_t tile_rows, int64_t tile_cols, double row_bytes,
                       int raster, int group, int64_t slots, int64_t lead, double l2_bytes)
{
    // Every tile of a wave streams its A row panel and B column panel through
    // K at about the same pace, so a panel shared by tiles of one wave is read
    // from DRAM once. Across waves a panel is still in L2 only if the previous
    // waves' panels fit (each wave starts again at k = 0, where a wave larger
    // than L2 has already been evicted): the store keeps whole waves, least
    // recently used first out, and forgets everything after a wave that does
    // not fit.
    const int64_t T = tiles_m * tiles_n;
    if (T <= 0 || slots < 1 || T > (int64_t(1) << 20))
        return 0.0;
    const double a_bytes = static_cast<double>(tile_rows) * row_bytes;
    const double b_bytes = static_cast<double>(tile_cols) * row_bytes;
    const int64_t P = tiles_m + tiles_n;  // panels: A rows 0..tiles_m-1, then B columns
    std::vector<int64_t> last(static_cast<size_t>(P), -1), in_wave(static_cast<size_t>(P), -1);
    std::vector<int64_t> wave_panels;
    double traffic = 0.0;
    int64_t wave = 0;
    for (int64_t t0 = 0; t0 < T; ++wave) {
        const int64_t t1 = std::min<int64_t>(T, t0 + (wave == 0 && lead > 0 ? lead : slots));
        wave_panels.clear();
        double foot = 0.0;
        for (int64_t t = t0; t < t1; ++t) {
            int64_t tm = 0, tn = 0;
            coord(t, tiles_m, tiles_n, raster, group, &tm, &tn);
            for (int64_t pnl : {tm, tiles_m + tn}) {
                if (in_wave[static_cast<size_t>(pnl)] == wave)
                    continue;
                in_wave[static_cast<size_t>(pnl)] = wave;
                wave_panels.push_back(pnl);
                const double b = pnl < tiles_m ? a_bytes : b_bytes;
                foot += b;
                if (last[static_cast<size_t>(pnl)] < 0)
                    traffic += b;
            }
        }
        if (foot > l2_bytes) {
            std::fill(last.begin(), last.end(), -1);
        } else {
            for (int64_t pnl : wave_panels)
                last[static_cast<size_t>(pnl)] = wave;
            // Evict the least recently used panels beyond the capacity.
            double cur = 0.0;
            std::vector<std::pair<int64_t, int64_t>> res;
            for (int64_t pnl = 0; pnl < P; ++pnl)
                if (last[static_cast<size_t>(pnl)] >= 0) {
                    cur += pnl < tiles_m ? a_bytes : b_bytes;
                    res.emplace_back(last[static_cast<size_t>(pnl)], pnl);
                }
            std::sort(res.begin(), res.end());
            for (const auto& r : res) {
                if (cur <= l2_bytes || r.first == wave)
                    break;
                cur -= r.second < tiles_m ? a_bytes : b_bytes;
                last[static_cast<size_t>(r.second)] = -1;
            }
        }
        t0 = t1;
    }
    return traffic;
}

bool parse_choice(const char* spec, Choice* out)
{
    Choice c{};
    c.splits = 1;
    if (!spec)
        return false;
    const int n = std::sscanf(spec, "%d,%d,%d,%d,%d", &c.bn, &c.cg, &c.raster, &c.group, &c.splits);
    if (n != 4 && n != 5)
        return false;
    if ((c.bn != 32 && c.bn != 64 && c.bn != 128 && c.bn != 256) || (c.cg != 1 && c.cg != 2) ||
        (c.raster != 0 && c.raster != 1) ||
        c.group < 1 || (c.cg == 2 && c.bn <= 64) || c.splits < 1 || c.splits > 16)
        return false;
    c.source = 2;
    *out = c;
    return true;
}

bool sk_layout(int64_t T, int64_t KB, int64_t G, int* sk_tiles, int* sk_w)
{
    if (KB < 1 || G < 2 || T <= G || T % G == 0)
        return false;
    // The partial wave alone, unless that would cut a tile into more than
    // about five pieces; then the last full wave joins it.
    int64_t sk = T % G;
    if (cdiv(sk * KB, G) * 4 < KB)
        sk += G;
    if (sk * KB > 0x7fffffffLL)
        return false;
    *sk_tiles = static_cast<int>(sk);
    *sk_w = static_cast<int>(cdiv(sk * KB, G));
    return true;
}

Choice select_config(int64_t M, int64_t N, int64_t K, int dt, int sm_count, bool tma_ok)
{
    // A table row's choice, fitted to the load path of this problem.
    auto from_row = [&](const TableRow& r, int source) {
        Choice c = r.c;
        c.source = source;
        if (c.splits < 1)
            c.splits = 1;
        if (!tma_ok && c.bn <= 64)
            c.bn = 128;
        if (!tma_ok) {
            // class-view tiles: 1-SM 128 or 256 columns, CTA-pair 256
            c.swap = 0;
            c.stages = 0;
            if (c.cg == 2)
                c.bn = 256;
        }
        return c;
    };
    for (const TableRow& r : kTable)
        if (r.dt == dt && r.M == M && r.N == N && r.K == K)
            return from_row(r, kSrcTable);
    // Power-of-two buckets: the nearest swept shape (in log2 distance) whose
    // M, N and K round up to the same powers of two and that took the same
    // load path. A swapped choice stays within M <= 128, where its kernels
    // tile M by 32 to 128 rows.
    if (M > 0 && N > 0 && K > 0) {
        const TableRow* best = nullptr;
        double best_d = 0.0;
        for (const TableRow& r : kTable) {
            if (r.dt != dt || r.M <= 0 || log2_ceil(r.M) != log2_ceil(M) || log2_ceil(r.N) != log2_ceil(N) ||
                log2_ceil(r.K) != log2_ceil(K) || tma_rows(r.K, r.N, dt) != tma_ok)
                continue;
            const double d = std::fabs(std::log2((double)r.M / M)) + std::fabs(std::log2((double)r.N / N)) +
                             std::fabs(std::log2((double)r.K / K));
            if (!best || d < best_d) {
                best = &r;
                best_d = d;
            }
        }
        if (best)
            return from_row(*best, kSrcBucket);
    }
    // Analytic rule, calibrated on the sweep: per-SM dense tensor rate
    // (bf16/fp16 8192 FLOP per clock, tf32 4096), a sustained operand fill
    // from L2 of about 64 bytes per clock per SM for TMA, about 22 bytes per
    // clock of HBM bandwidth per SM (6.7 TB/s over 152 SMs at ~2 GHz), and a
    // fixed cost per wave (prologue, pipeline fill, final epilogue). Rows that
    // TMA cannot address directly (tma_ok false) take the class-view kernels,
    // also TMA-fed: 1-SM 128 or 256 columns, or CTA-pair 256; B is first
    // packed into aligned rows when its own are not (one read and one write
    // of B more).
    const double es = dt == 0 ? 4.0 : 2.0;
    const double flop_clk = dt == 0 ? 4096.0 : 8192.0;
    const double fill_clk = 64.0;
    const double hbm_clk = 22.0 * sm_count;
    const double wave_cost = 6000.0;
    const double pack = !tma_ok && (N * static_cast<int64_t>(es)) % 16 != 0 ? 2.0 * es * (double)(K * N) / hbm_clk : 0.0;
    const double hbm = (es * (double)(M * K + K * N) + 8.0 * (double)(M * N)) / hbm_clk + pack;
    struct Cand { int bn, cg, swap; };
    // Tiles of a candidate: 128 x cta_group rows by bn columns of C, or,
    // swapped, 128 columns by bn rows.
    auto tiles_of = [&](int bn, int cg, int swap) {
        return swap ? cdiv(N, 128) * cdiv(M, bn) : cdiv(M, 128 * cg) * cdiv(N, bn);
    };
    const Cand cands[] = {{256, 2, 0}, {128, 2, 0}, {256, 1, 0}, {128, 1, 0}, {64, 1, 0}};
    double best_t = 1e300;
    Choice best{256, 1, 0, 8, 0};
    for (const Cand& cd : cands) {
        if (!tma_ok && (cd.bn == 64 || cd.swap || (cd.cg == 2 && cd.bn != 256)))
            continue;
        if (cd.cg == 2 && M <= 128)
            continue;  // a CTA pair would leave its second 128 rows empty
        const int64_t tiles = tiles_of(cd.bn, cd.cg, cd.swap);
        const int64_t slots = std::max<int64_t>(1, sm_count / cd.cg);
        const int64_t waves = cdiv(tiles, slots);
        // Per CTA: its MMA share and the bytes it loads per unit of K.
        const double mma = 2.0 * 128.0 * cd.bn * K / flop_clk;
        const double fill = (128.0 + cd.bn / cd.cg) * es * K / fill_clk;
        const double t = std::max(waves * (std::max(mma, fill) + wave_cost) + pack, hbm);
        // Prefer the larger tile unless the smaller is clearly faster.
        if (t < best_t * 0.97) {
            best_t = t;
            best.bn = cd.bn;
            best.cg = cd.cg;
            best.swap = cd.swap;
        }
    }
    // At most 32 rows: 128-row tiles of C would be three-quarters empty, so
    // exchange the operands' roles and tile C^T, 128 columns by 32 rows. (Such
    // shapes are HBM-bound either way; measured, the swap was 0-6% faster at
    // 16 and 32 rows and 0-5% slower at 64.)
    if (tma_ok && M <= 32) {
        best.bn = 32;
        best.cg = 1;
        best.swap = 1;
    }
    best.raster = 0;
    best.group = best.cg == 2 ? 4 : 8;
    best.source = kSrcRule;
    best.splits = 1;
    best.stages = 0;
    // beta != 0: fetching C through the operand ring pays when C is a large
    // share of a tile's traffic (short K); with a long K loop the epilogue's
    // own C loads hide behind the next tile's main loop, and the ring stages
    // that C would hold are worth more to the operands.
    best.cload = cdiv(K, dt == 0 ? 32 : 64) > 32 ? 1 : 0;
    // Split K when the chosen tiles would leave most SMs idle and K is long:
    // each split needs at least 16 k-blocks, and the fixed-order reduction
    // (S + 2 floats of traffic per output) plus its launch must pay off.
    {
        const int64_t ctas = tiles_of(best.bn, best.cg, best.swap) * best.cg;
        const int64_t kb = cdiv(K, dt == 0 ? 32 : 64);
        int s = 1;
        while (s < 8 && ctas * s * 2 <= sm_count && kb / (s * 2) >= 16)
            s *= 2;
        if (s > 1) {
            const double mma = 2.0 * 128.0 * best.bn * K / flop_clk;
            const double fill = (128.0 + best.bn / best.cg) * es * K / fill_clk;
            const double t1 = std::max(mma, fill) + wave_cost;
            const double ts = std::max(mma, fill) / s + wave_cost + 6000.0 + (s + 2.0) * 4.0 * (double)(M * N) / hbm_clk;
            if (ts < 0.8 * t1)
                best.splits = s;
        }
    }
    // Stream-K when more than one wave of tiles ends in a partial one whose
    // idle share is worth at least 3% of the run, and K is long enough for
    // the fix-up of a split tile (one partial tile written and read per
    // contributor) to be small against a tile's K loop.
    // (Not for class-view tiles, tma_ok false: their stream-K pieces end in the
    // row-store epilogue, measured 1.4-1.7x slower than whole tiles at
    // (8191, 4097, 2049).)
    if (best.splits == 1 && tma_ok) {
        const int64_t tiles = tiles_of(best.bn, best.cg, best.swap);
        const int64_t slots = std::max<int64_t>(1, sm_count / best.cg);
        const int64_t kb = cdiv(K, dt == 0 ? 32 : 64);
        const double f = static_cast<double>(tiles % slots) / static_cast<double>(slots);
        const double idle = f > 0.0 ? (1.0 - f) / static_cast<double>(cdiv(tiles, slots)) : 0.0;
        best.sk = tiles > slots && idle >= 0.03 && kb >= 32 ? 1 : 0;
    }
    // Raster order and group: the least operand traffic from DRAM in the model
    // above, with an effective L2 of 60 MB (calibrated on ncu's DRAM bytes of
    // four stream-K squares and tails; the rest of the 129 MB holds C's
    // write-back, the partial tiles and lines duplicated across the two dies).
    // Ties keep the default, then the smaller group.
    {
        const int64_t rows = best.swap ? N : M, cols = best.swap ? M : N;
        const int64_t tile_rows = best.swap ? 128 : 128 * best.cg, tile_cols = best.bn;
        const int64_t tiles_m = cdiv(rows, tile_rows), tiles_n = cdiv(cols, tile_cols);
        const int64_t slots = std::max<int64_t>(1, sm_count / best.cg);
        const int64_t kb = cdiv(K, dt == 0 ? 32 : 64);
        int64_t lead = 0;
        if (best.sk) {
            int skt = 0, skw = 0;
            if (sk_layout(tiles_m * tiles_n, kb, slots, &skt, &skw))
                lead = skt;
        }
        const double row_bytes = es * static_cast<double>(K);
        double t_best = operand_traffic(tiles_m, tiles_n, tile_rows, tile_cols, row_bytes, best.raster, best.group,
                                        slots, lead, kL2Effective);
        for (int raster : {0, 1})
            for (int group : {1, 2, 4, 8, 16}) {
                const double t = operand_traffic(tiles_m, tiles_n, tile_rows, tile_cols, row_bytes, raster, group,
                                                 slots, lead, kL2Effective);
                if (t < t_best * 0.98) {
                    t_best = t;
                    best.raster = raster;
                    best.group = group;
                }
            }
    }
    return best;
}

}  // namespace sat
