// Host side of the C ABI declared in include/gemm.h: plan creation (device
// checks, dispatcher, kernel preparation), tensor-map encoding and launch.
#include "gemm.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <new>

#include "dispatch.h"
#include "registry.h"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int elem_size(int dt) { return dt == sat::kDtTF32 ? 4 : 2; }

const char* dt_name(int dt) { return dt == 0 ? "tf32" : dt == 1 ? "bf16" : "fp16"; }

// 2-D row-major tensor map with a 128-byte-swizzled box of box_inner x
// box_outer elements; out-of-bounds elements of a box read as zero.
int encode_2d(CUtensorMap* map, int dt, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer, CUtensorMapSwizzle swizzle, uint64_t ld = 0)
{
    const CUtensorMapDataType t = dt == sat::kDtTF32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                  : dt == sat::kDtBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const int r = sat::encode_map(map, t, elem_size(dt), ptr, inner, outer, ld ? ld : inner, box_inner, box_outer,
                                  swizzle);
    if (r == -1)
        return fail(GEMM_ERR_LAUNCH, "cuTensorMapEncodeTiled is not available from the driver");
    if (r != 0)
        return fail(GEMM_ERR_LAUNCH, "cuTensorMapEncodeTiled failed (%d)", r);
    return 0;
}

int cuda_fail(cudaError_t e, const char* what)
{
    return fail(GEMM_ERR_LAUNCH, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace

namespace sat {
void set_last_error(const char* msg)
{
    std::snprintf(g_err, sizeof g_err, "%s", msg);
}

int fail_with(int code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}
}  // namespace sat

namespace {

// Device scratch that the runs of a split-K or stream-K plan write: the
// split-K partial tiles, or the stream-K partial tiles, counters and slot
// ticket. One set per stream the plan runs on, so that runs on different
// streams never share them; the stream's own order keeps runs on one stream
// apart. At most kMaxScratch sets per plan: past that, a new stream takes
// over the set used least recently, behind that set's last run (a wait on
// the GPU for the event recorded after it, not on the host).
struct Scratch {
    unsigned long long stream_id = 0;  // cudaStreamGetId of the stream that uses it
    float* ws = nullptr;               // split-K: splits x ws_rows x N floats
    CUtensorMap tmW{};                 // ws for the bulk-store epilogue
    bool ws_tma = false;
    float* sk_ws = nullptr;            // stream-K: one 128 x bn float partial tile per CTA
    unsigned* sk_flags = nullptr;      // stream-K: one counter per CTA, then the ticket counter
    unsigned epoch = 0;                // stream-K launches on these counters since they were cleared
    unsigned long long sk_sig = 0;     // the stream-K layout those launches used
    void* bpack = nullptr;             // B in rows of whole 128-byte lines (K x ldb_pack elements), when its own rows are not TMA-addressable
    cudaEvent_t done = nullptr;        // recorded after each run that used this set
    unsigned long long last_use = 0;
    // gemm_run_host in row blocks: copy streams (host to device, device to
    // host) and their events (start, one per block copied in, one per block
    // computed, end).
    cudaStream_t cp_in = nullptr, cp_out = nullptr;
    cudaEvent_t hev[2 + 2 * 8] = {};
};
constexpr int kMaxScratch = 8;
// Row blocks of a pipelined gemm_run_host: at most 8 (the last block's GEMM
// and copy out are the part that overlaps nothing), of at least 512 rows.
constexpr int kHostBlocks = 8;
constexpr int64_t kHostMinRows = 512;
static_assert(sizeof(Scratch::hev) / sizeof(cudaEvent_t) == 2 + 2 * kHostBlocks, "one event per block copied in and computed");
constexpr int kTicketPad = 32;  // the ticket counter sits 128 bytes past the last CTA counter

}  // namespace

struct gemm_plan {
    int64_t M = 0, N = 0, K = 0;
    int dt = 0;
    int device = 0;
    int sm_count = 0;
    bool trans_a = false, trans_b = false;  // A stored K x M, B stored N x K
    int c_half = 0;                         // element type of C: 0 fp32, 1 bf16, 2 fp16
    sat::Choice choice{};
    bool force_plain = false;
    bool alt_k = true;    // alternate waves run through K in opposite directions
    bool c_ring = false;  // beta != 0: the producer fetches C through the operand ring
    const sat::KernelEntry* tma = nullptr;    // null when the strides rule out TMA
    const sat::KernelEntry* plain = nullptr;  // 1-SM plain-load variant (misaligned pointers)
    const sat::KernelEntry* plain_strided = nullptr;  // the same, for row strides other than K and N
    // Class-view kernel for operand rows that TMA cannot address directly
    // (untransposed plans): A through one tensor map per residue class of row
    // index, B aligned or packed into the stream's scratch (ldb_pack).
    const sat::KernelEntry* cls = nullptr;
    int64_t slots_cls = 0, ldb_pack = 0;
    int grid_tma = 0, grid_plain = 0;
    // Error word in host-mapped pinned memory: kernels OR bits into it through
    // d_err; the host reads h_err without synchronising.
    uint32_t* h_err = nullptr;
    uint32_t* d_err = nullptr;
    // Split-K: `splits` slices of `ws_rows` x N floats, reduced in fixed order
    // into C (the slices live in the per-stream scratch).
    int splits = 1, kb_per_split = 0, ws_rows = 0;
    // Stream-K (the choice's sk): layout, and per-stream scratch of one
    // 128 x BN partial tile and one counter per CTA.
    int sk_tiles = 0, sk_w = 0, sk_ctas = 0, sk_bn = 0;
    mutable std::mutex scratch_mu;
    mutable Scratch scratch[kMaxScratch];
    mutable int n_scratch = 0;
    mutable unsigned long long use_clock = 0;
    unsigned long long timeout_ns = 2000000000ull;
    char desc[256] = "";
    mutable std::mutex mu;
    // Plans for the row blocks of a pipelined gemm_run_host (rows of every
    // block but the last, and of the last), made by its first such run.
    mutable gemm_plan* host_plan[2] = {nullptr, nullptr};
    mutable int64_t host_rows[2] = {0, 0};
    mutable const void* map_A = nullptr;
    mutable const void* map_B = nullptr;
    mutable const void* map_C = nullptr;
    mutable int64_t map_lda = 0, map_ldb = 0, map_ldc = 0;
    mutable CUtensorMap tmA{}, tmB{}, tmC{};
    // Class views of A (for the A pointer and stride they were made for).
    mutable const void* cls_A = nullptr;
    mutable int64_t cls_lda = 0;
    mutable int cls_n = 0;
    mutable int cls_shift[sat::kMaxClasses] = {}, cls_rows[sat::kMaxClasses] = {};
    mutable CUtensorMap tmCls[sat::kMaxClasses];
    mutable const void* cls_B = nullptr;
    mutable int64_t cls_ldb = 0;
    mutable CUtensorMap tmClsB{};
};

namespace {

// CTA slots (single CTAs, or pairs) that can be resident at once.
int64_t slots_for(const gemm_plan* p, const sat::KernelEntry* e)
{
    int64_t slots = p->sm_count / e->cg;
    if (e->cg == 2) {
        // Not every SM need be able to pair with a neighbour: ask the
        // occupancy calculator how many CTA pairs can be resident at once.
        const int n = e->max_clusters();
        if (n > 0 && n < slots)
            slots = n;
    }
    return slots < 1 ? 1 : slots;
}

int grid_for(const gemm_plan* p, const sat::KernelEntry* e)
{
    int64_t tm = 0, tn = 0;
    sat::tile_grid(e, p->M, p->N, &tm, &tn);
    const int64_t tiles = tm * tn * p->splits;
    const int64_t slots = slots_for(p, e);
    return static_cast<int>((tiles < slots ? tiles : slots) * e->cg);
}

gemm_plan* create(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, const char* config, bool trans_a = false,
                  bool trans_b = false, int c_type = 0)
{
    if (c_type < 0 || c_type > 2) {
        fail(GEMM_ERR_ARG, "unknown C type %d", c_type);
        return nullptr;
    }
    g_err[0] = '\0';
    const int dt = static_cast<int>(dtype);
    if (M < 0 || N < 0 || K < 0 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31)) {
        fail(GEMM_ERR_ARG, "dimensions must be in [0, 2^31): M=%lld N=%lld K=%lld", (long long)M, (long long)N,
             (long long)K);
        return nullptr;
    }
    if (dt < 0 || dt > 2) {
        fail(GEMM_ERR_ARG, "unknown dtype %d", dt);
        return nullptr;
    }
    int dev = 0, major = 0, minor = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        cuda_fail(e, "querying the device");
        return nullptr;
    }
    if (major != 10 || minor != 3) {
        fail(GEMM_ERR_ARCH, "device %d is compute capability %d.%d; this library is built for sm_103a only", dev,
             major, minor);
        return nullptr;
    }
    gemm_plan* p = new (std::nothrow) gemm_plan;
    if (!p) {
        fail(GEMM_ERR_NOMEM, "out of host memory");
        return nullptr;
    }
    p->M = M;
    p->N = N;
    p->K = K;
    p->dt = dt;
    p->device = dev;
    p->sm_count = sms;
    p->trans_a = trans_a;
    p->trans_b = trans_b;
    p->c_half = c_type;
    const int64_t es = elem_size(dt);
    // Dense row strides that TMA can describe. Transposed operands are read
    // by TMA only, so their plans assume it (gemm_run_ex checks each call).
    const bool trans = trans_a || trans_b;
    const bool tma_ok = trans || ((K * es) % 16 == 0 && (N * es) % 16 == 0);

    const char* source = "rule";
    if (config && config[0]) {
        char head[64];
        std::snprintf(head, sizeof head, "%s", config);
        // Optional tags after the numbers, in any order: ",cload" (the
        // epilogue loads C itself), ",sk" (stream-K), ",plain" (plain-load
        // producer). Each is looked up first; the numbers end at the first.
        char* tag[6] = {std::strstr(head, ",cload"), std::strstr(head, ",sk"), std::strstr(head, ",plain"),
                        std::strstr(head, ",swap"), std::strstr(head, ",st"), std::strstr(head, ",fwd")};
        // ",fwd": every wave runs through K forwards (no alternating direction).
        p->alt_k = tag[5] == nullptr;
        const bool cload = tag[0] != nullptr, sk = tag[1] != nullptr, swap = tag[3] != nullptr;
        p->force_plain = tag[2] != nullptr;
        // ",st<n>": a ring of n stages (a compiled depth of the TMA kernel).
        int stages = 0;
        if (tag[4] && std::sscanf(tag[4] + 3, "%d", &stages) != 1)
            stages = -1;
        for (char* t : tag)
            if (t)
                *t = '\0';
        if (!sat::parse_choice(head, &p->choice)) {
            fail(GEMM_ERR_ARG,
                 "bad configuration \"%s\" (want \"bn,cg,raster,group[,splits][,cload][,sk][,swap][,plain]\")",
                 config);
            delete p;
            return nullptr;
        }
        p->choice.cload = cload ? 1 : 0;
        p->choice.sk = sk ? 1 : 0;
        p->choice.swap = swap ? 1 : 0;
        p->choice.stages = stages;
        if (stages < 0) {
            fail(GEMM_ERR_ARG, "bad configuration \"%s\" (\",st\" wants a stage count)", config);
            delete p;
            return nullptr;
        }
        if (swap && (p->choice.cg != 1 || p->choice.bn == 256)) {
            fail(GEMM_ERR_ARG, "bad configuration \"%s\" (a swapped tile is 1-SM with bn 32, 64 or 128)", config);
            delete p;
            return nullptr;
        }
        source = "forced";
    } else {
        p->choice = sat::select_config(M, N, K, dt, sms, tma_ok);
        source = p->choice.source == sat::kSrcTable ? "table" : p->choice.source == sat::kSrcBucket ? "bucket" : "rule";
    }
    if (trans) {
        // Transposed layouts come as 1-SM 128 x 128 and 128 x 256 tiles and
        // 256 x 256 CTA-pair tiles, unswapped, with TMA loads only.
        sat::Choice& cc = p->choice;
        cc.swap = 0;
        cc.bn = cc.cg == 2 ? 256 : (cc.bn < 256 ? 128 : 256);
        if (p->force_plain) {
            fail(GEMM_ERR_ARG, "transposed operands have no plain-load kernel");
            delete p;
            return nullptr;
        }
    }
    const sat::Choice& c = p->choice;
    const int tma_kind = trans_a && trans_b ? sat::kProdTT
                         : trans_a          ? sat::kProdTN
                         : trans_b          ? sat::kProdNT
                         : c.swap           ? sat::kProdSwap
                                            : sat::kProdTMA;
    if (tma_ok && !p->force_plain) {
        p->tma = sat::find_entry(dt, c.bn, c.cg, tma_kind, tma_kind == sat::kProdTMA ? c.stages : 0);
        if (!p->tma) {
            fail(GEMM_ERR_ARG, "no compiled TMA kernel for bn=%d cg=%d stages=%d in this layout", c.bn, c.cg,
                 c.stages);
            delete p;
            return nullptr;
        }
    }
    // B's rows not 16-byte multiples (N) while A's are (K): the TMA kernel,
    // with B packed into aligned rows at run time, where the choice has one.
    if (!tma_ok && !trans && !p->force_plain && !c.swap && (K * es) % 16 == 0)
        p->tma = sat::find_entry(dt, c.bn, c.cg, sat::kProdTMA, c.stages);
    if (!trans) {
        p->plain = sat::find_entry(dt, c.bn < 128 ? 128 : c.bn, 1, sat::kProdPlain);
        p->plain_strided = sat::find_entry(dt, c.bn < 128 ? 128 : c.bn, 1, sat::kProdPlainStrided);
        if (!p->plain || !p->plain_strided) {
            fail(GEMM_ERR_ARG, "no compiled plain-load kernel for bn=%d", c.bn);
            delete p;
            return nullptr;
        }
    }
    if (!trans && !p->force_plain) {
        // The class-view kernel serves operand rows that TMA cannot address:
        // the choice's tile where one is compiled (1-SM 128 or 256 columns,
        // CTA-pair 256).
        const int bn = c.cg == 2 ? 256 : (c.bn < 128 ? 128 : c.bn);
        p->cls = sat::find_entry(dt, bn, c.cg, sat::kProdClassA);
        if (p->cls)
            p->slots_cls = slots_for(p, p->cls);

        // Packed rows of B span an odd number of whole 128-byte lines: each
        // TMA box row is then one line (rows only 16-byte aligned straddle
        // two, and five 32-byte sectors), and rows do not repeat at a
        // power-of-two stride. At bf16 (8191, 4097, 2049) the packed B read
        // with 4104-element rows cost 16 us more than with 4160.
        int64_t lines = (N * es + 127) / 128;
        if (lines % 2 == 0)
            ++lines;
        p->ldb_pack = lines * 128 / es;
    }
    for (const sat::KernelEntry* k : {p->tma, p->plain, p->plain_strided, p->cls}) {
        if (!k)
            continue;
        e = k->prepare();
        if (e != cudaSuccess) {
            cuda_fail(e, "setting the kernel's shared-memory limit");
            delete p;
            return nullptr;
        }
    }
    // Split-K over this plan's tiles (TMA and plain-load variants share the
    // tile N, and both use single-CTA row tiles of 128 when plain).
    const int bk = (p->tma ? p->tma : p->plain)->bk;
    const int64_t num_kb = (K + bk - 1) / bk;
    p->splits = c.splits > 1 && num_kb > 1 ? c.splits : 1;
    if (p->splits > num_kb)
        p->splits = static_cast<int>(num_kb);
    p->kb_per_split = static_cast<int>((num_kb + p->splits - 1) / p->splits);
    if (p->splits > 1)  // no empty split
        p->splits = static_cast<int>((num_kb + p->kb_per_split - 1) / p->kb_per_split);
    if (p->tma)
        p->grid_tma = grid_for(p, p->tma);
    if (p->plain)
        p->grid_plain = grid_for(p, p->plain);
    e = cudaHostAlloc(reinterpret_cast<void**>(&p->h_err), 64, cudaHostAllocMapped);
    if (e == cudaSuccess) {
        *reinterpret_cast<volatile uint32_t*>(p->h_err) = 0;
        e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&p->d_err), p->h_err, 0);
    }
    if (p->splits > 1)
        p->ws_rows = static_cast<int>((M + 255) / 256 * 256);
    // Stream-K (TMA path, unsplit): every slot runs, whatever the tile count.
    if (e == cudaSuccess && c.sk && p->tma && p->splits == 1) {
        const sat::KernelEntry* t = p->tma;
        int64_t tm = 0, tn = 0;
        sat::tile_grid(t, M, N, &tm, &tn);
        const int64_t tiles = tm * tn;
        const int64_t slots = slots_for(p, t);
        if (sat::sk_layout(tiles, num_kb, slots, &p->sk_tiles, &p->sk_w)) {
            p->sk_ctas = static_cast<int>(slots * t->cg);
            p->sk_bn = t->bn;
            p->grid_tma = p->sk_ctas;
        }
    }
    // Class-view runs lay out stream-K per run (their tiles depend on A's
    // alignment); size the scratch for their grid too.
    if (p->cls && c.sk && p->splits == 1) {
        p->sk_ctas = std::max<int>(p->sk_ctas, static_cast<int>(p->slots_cls * p->cls->cg));
        p->sk_bn = std::max(p->sk_bn, p->cls->bn);
    }
    if (e != cudaSuccess) {
        cuda_fail(e, "allocating the host-mapped error word");
        if (p->h_err)
            cudaFreeHost(p->h_err);
        delete p;
        return nullptr;
    }
    if (const char* t = std::getenv("SAT_GEMM_WAIT_TIMEOUT_MS")) {
        const long long ms = std::atoll(t);
        if (ms > 0)
            p->timeout_ns = static_cast<unsigned long long>(ms) * 1000000ull;
    }
    const sat::KernelEntry* k = p->tma ? p->tma : p->cls ? p->cls : p->plain;
    p->c_ring = !c.cload && p->tma && p->tma->c_ring && p->splits == 1 && p->sk_tiles == 0 && p->c_half == 0;
    char sk_desc[48] = "";
    if (p->sk_tiles)
        std::snprintf(sk_desc, sizeof sk_desc, " sk%d/%d", p->sk_tiles, p->sk_w);
    std::snprintf(p->desc, sizeof p->desc, "%s m%lld n%lld k%lld: bn%d cg%d st%d %s raster%d g%d s%d grid%d %s%s%s%s%s%s",
                  dt_name(dt), (long long)M, (long long)N, (long long)K, k->bn, k->cg, k->stages,
                  p->tma ? "tma" : p->cls ? "cls" : "plain", c.raster, c.group, p->splits,
                  p->tma ? p->grid_tma : p->cls ? static_cast<int>(p->slots_cls * p->cls->cg) : p->grid_plain,
                  source, p->c_ring ? " cring" : "", sk_desc, p->tma && p->tma->prod == sat::kProdSwap ? " swap" : "",
                  trans_a ? " ta" : "", trans_b ? " tb" : "");
    if (!p->alt_k)
        std::snprintf(p->desc + std::strlen(p->desc), sizeof p->desc - std::strlen(p->desc), " fwd");
    if (c_type)
        std::snprintf(p->desc + std::strlen(p->desc), sizeof p->desc - std::strlen(p->desc), " c%s",
                      c_type == 1 ? "bf16" : "fp16");
    return p;
}

}  // namespace

namespace {

void free_scratch(Scratch& s)
{
    for (void* d : {static_cast<void*>(s.ws), static_cast<void*>(s.sk_ws), static_cast<void*>(s.sk_flags), s.bpack})
        if (d)
            cudaFree(d);
    if (s.done)
        cudaEventDestroy(s.done);
    for (cudaEvent_t ev : s.hev)
        if (ev)
            cudaEventDestroy(ev);
    for (cudaStream_t st : {s.cp_in, s.cp_out})
        if (st)
            cudaStreamDestroy(st);
    s = Scratch{};
}

size_t sk_flag_bytes(const gemm_plan* p)
{
    return static_cast<size_t>(p->sk_ctas + kTicketPad) * sizeof(unsigned);
}

// The scratch set of `stream` (p->scratch_mu held): this stream's own, a new
// one, or the least recently used one taken over behind its last run. A new
// set's counters are cleared on `stream`, ahead of the run.
int acquire_scratch(const gemm_plan* p, cudaStream_t stream, bool want_pack, Scratch** out)
{
    unsigned long long id = 0;
    cudaError_t e = cudaStreamGetId(stream, &id);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaStreamGetId");
    Scratch* hit = nullptr;
    for (int i = 0; i < p->n_scratch && !hit; ++i)
        if (p->scratch[i].stream_id == id)
            hit = &p->scratch[i];
    if (!hit && p->n_scratch < kMaxScratch) {
        Scratch& s = p->scratch[p->n_scratch];
        e = cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming);
        if (e == cudaSuccess && p->splits > 1) {
            const size_t bytes =
                static_cast<size_t>(p->splits) * p->ws_rows * static_cast<size_t>(p->N) * sizeof(float);
            e = cudaMalloc(&s.ws, bytes);
            if (e == cudaSuccess && (p->N * 4) % 16 == 0 &&
                encode_2d(&s.tmW, sat::kDtTF32, s.ws, p->N, static_cast<uint64_t>(p->splits) * p->ws_rows, 32u, 32u,
                          CU_TENSOR_MAP_SWIZZLE_128B) == 0)
                s.ws_tma = true;
        }
        if (e == cudaSuccess && p->sk_ctas > 0) {
            e = cudaMalloc(&s.sk_ws, static_cast<size_t>(p->sk_ctas) * 128 * p->sk_bn * sizeof(float));
            if (e == cudaSuccess)
                e = cudaMalloc(&s.sk_flags, sk_flag_bytes(p));
            if (e == cudaSuccess)
                e = cudaMemsetAsync(s.sk_flags, 0, sk_flag_bytes(p), stream);
        }
        if (e != cudaSuccess) {
            free_scratch(s);
            return fail(e == cudaErrorMemoryAllocation ? GEMM_ERR_NOMEM : GEMM_ERR_LAUNCH,
                        "preparing this stream's scratch: %s", cudaGetErrorString(e));
        }
        s.stream_id = id;
        ++p->n_scratch;
        hit = &s;
    }
    if (!hit) {
        Scratch* v = &p->scratch[0];
        for (int i = 1; i < p->n_scratch; ++i)
            if (p->scratch[i].last_use < v->last_use)
                v = &p->scratch[i];
        e = cudaStreamWaitEvent(stream, v->done, 0);
        if (e != cudaSuccess)
            return cuda_fail(e, "ordering this stream behind the scratch's last run");
        v->stream_id = id;
        hit = v;
    }
    if (want_pack && !hit->bpack) {
        const size_t bytes = static_cast<size_t>(p->K) * static_cast<size_t>(p->ldb_pack) * elem_size(p->dt);
        e = cudaMalloc(&hit->bpack, bytes);
        if (e != cudaSuccess) {
            hit->bpack = nullptr;
            return fail(e == cudaErrorMemoryAllocation ? GEMM_ERR_NOMEM : GEMM_ERR_LAUNCH,
                        "allocating this stream's aligned copy of B: %s", cudaGetErrorString(e));
        }
    }
    hit->last_use = ++p->use_clock;
    *out = hit;
    return GEMM_OK;
}

int run_impl(const gemm_plan* p, const void* A, int64_t lda, const void* B, int64_t ldb, void* Cv, int64_t ldc,
             float alpha, float beta, void* cuda_stream)
{
    float* C = static_cast<float*>(Cv);  // fp32, or 16-bit elements when the plan's C type says so
    if (!p)
        return fail(GEMM_ERR_ARG, "plan is NULL");
    if (p->M == 0 || p->N == 0)
        return GEMM_OK;
    if (lda >= (int64_t(1) << 31) || ldb >= (int64_t(1) << 31) || ldc >= (int64_t(1) << 31))
        return fail(GEMM_ERR_ARG, "leading dimensions must be below 2^31");
    if ((p->K > 0 && (lda < (p->trans_a ? p->M : p->K) || ldb < (p->trans_b ? p->K : p->N))) || ldc < p->N)
        return fail(GEMM_ERR_ARG, "leading dimension too small (lda %lld, ldb %lld, ldc %lld)", (long long)lda,
                    (long long)ldb, (long long)ldc);
    if (!C)
        return fail(GEMM_ERR_ARG, "C is NULL");
    if (reinterpret_cast<uintptr_t>(C) % (p->c_half ? 2 : 4) != 0)
        return fail(GEMM_ERR_ALIGN, "C must be aligned to its element size");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev != p->device)
        return fail(GEMM_ERR_ARG, "plan was made for device %d but device %d is current", p->device, dev);
    // A kernel of this plan that gave up a bounded wait set the host-mapped
    // error word: report it here, before enqueueing more work.
    if (*reinterpret_cast<volatile uint32_t*>(p->h_err) != 0)
        return fail(GEMM_ERR_TIMEOUT,
                    "an earlier run of this plan gave up a bounded wait (its C is incomplete); nothing was enqueued; "
                    "gemm_plan_status clears the condition");
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    if (p->K == 0 || alpha == 0.0f) {
        e = sat::launch_scale(C, p->c_half, p->M, p->N, ldc, beta, stream);
        return e == cudaSuccess ? GEMM_OK : cuda_fail(e, "launching the beta-scale kernel");
    }
    if (!A || !B)
        return fail(GEMM_ERR_ARG, "A or B is NULL");
    const uintptr_t es = static_cast<uintptr_t>(elem_size(p->dt));
    if (reinterpret_cast<uintptr_t>(A) % es || reinterpret_cast<uintptr_t>(B) % es)
        return fail(GEMM_ERR_ALIGN, "A and B must be aligned to their %d-byte element size", (int)es);
    // TMA needs 16-byte aligned bases and row strides.
    const int64_t es64 = static_cast<int64_t>(es);
    const bool a_rows_ok = reinterpret_cast<uintptr_t>(A) % 16 == 0 && (lda * es64) % 16 == 0;
    const bool b_rows_ok = reinterpret_cast<uintptr_t>(B) % 16 == 0 && (ldb * es64) % 16 == 0;
    // B's rows, where TMA cannot address them, are packed into this
    // stream's aligned copy first (untransposed B only).
    const bool b_pack_ok = !p->trans_b && p->ldb_pack > 0;
    const bool use_tma = p->tma && a_rows_ok && (b_rows_ok || b_pack_ok);
    // Otherwise (untransposed plans) the class-view kernel: A through one
    // tensor map per residue class of row index, B as it lies or packed.
    const bool use_cls = !use_tma && p->cls != nullptr;
    if (!use_tma && !use_cls && !p->plain)
        return fail(GEMM_ERR_ALIGN,
                    "transposed operands are read by TMA only: A and B must be 16-byte aligned with row strides "
                    "that are multiples of 16 bytes");
    const bool dense = lda == p->K && ldb == p->N;
    const sat::KernelEntry* k = use_tma ? p->tma : use_cls ? p->cls : dense ? p->plain : p->plain_strided;

    sat::GemmArgs a{};
    a.M = static_cast<int>(p->M);
    a.N = static_cast<int>(p->N);
    a.K = static_cast<int>(p->K);
    a.A = A;
    a.B = B;
    a.C = C;
    a.lda = static_cast<int>(lda);
    a.ldb = static_cast<int>(ldb);
    a.ldc = static_cast<int>(ldc);
    a.c_half = p->c_half;
    a.alpha = alpha;
    a.beta = beta;
    int64_t tiles_m = 0, tiles_n = 0;
    sat::tile_grid(k, p->M, p->N, &tiles_m, &tiles_n);
    a.num_kb = static_cast<int>((p->K + k->bk - 1) / k->bk);
    int splits = p->splits, kbps = p->kb_per_split;
    if (use_cls) {
        // Residue classes of A's rows: row m starts (A + m * lda * es) mod 16
        // bytes past a 16-byte boundary, which repeats with period P. Class r
        // (rows r + P*y) is read from a view starting that many bytes earlier,
        // so every class's view rows are 16-byte aligned. Output tiles take
        // 128 x cta_group view rows of one class; K runs over the views'
        // extra leading elements too.
        std::lock_guard<std::mutex> lock(p->mu);
        if (p->cls_A != A || p->cls_lda != lda) {
            const int64_t rb = lda * es64;
            int g = static_cast<int>(rb % 16);
            int P = 16;
            while (g && P > 1 && g % 2 == 0 && P % 2 == 0) {
                g /= 2;
                P /= 2;
            }
            if (g == 0)
                P = 1;
            const CUtensorMapDataType t = p->dt == sat::kDtTF32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                          : p->dt == sat::kDtBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
            for (int r = 0; r < P; ++r) {
                const uintptr_t start = reinterpret_cast<uintptr_t>(A) + static_cast<uintptr_t>(r * rb);
                const int delta = static_cast<int>(start % 16);
                const int64_t rows = r < p->M ? (p->M - r + P - 1) / P : 0;
                p->cls_shift[r] = delta / static_cast<int>(es);
                p->cls_rows[r] = static_cast<int>(rows);
                // A class without rows reads class 0's view (its tiles store nothing).
                const int src = rows > 0 ? r : 0;
                const uintptr_t sstart = reinterpret_cast<uintptr_t>(A) + static_cast<uintptr_t>(src * rb);
                const int sdelta = static_cast<int>(sstart % 16);
                const int64_t srows = (p->M - src + P - 1) / P;
                const int rc = sat::encode_map(&p->tmCls[r], t, static_cast<int>(es),
                                               reinterpret_cast<const void*>(sstart - sdelta),
                                               static_cast<uint64_t>(p->K + sdelta / static_cast<int>(es)),
                                               static_cast<uint64_t>(srows), static_cast<uint64_t>(P * lda),
                                               static_cast<uint32_t>(k->bk), 128u, CU_TENSOR_MAP_SWIZZLE_128B);
                if (rc) {
                    p->cls_A = nullptr;
                    return fail(GEMM_ERR_LAUNCH, "cuTensorMapEncodeTiled failed for a class view of A (%d)", rc);
                }
            }
            p->cls_n = P;
            p->cls_A = A;
            p->cls_lda = lda;
        }
        a.a_classes = p->cls_n;
        int smax = 0;
        for (int r = 0; r < p->cls_n; ++r) {
            a.a_shift[r] = p->cls_shift[r];
            a.a_rows[r] = p->cls_rows[r];
            smax = std::max(smax, p->cls_shift[r]);
        }
        const int64_t per_class = (p->M + p->cls_n - 1) / p->cls_n;
        tiles_m = p->cls_n * ((per_class + 128 * k->cg - 1) / (128 * k->cg));
        a.num_kb = static_cast<int>((p->K + smax + k->bk - 1) / k->bk);
        if (splits > 1) {
            // The same slices of the workspace, over the views' k-blocks.
            kbps = (a.num_kb + splits - 1) / splits;
            splits = (a.num_kb + kbps - 1) / kbps;
        }
    }
    a.tiles_m = static_cast<int>(tiles_m);
    a.tiles_n = static_cast<int>(tiles_n);
    a.splits = splits;
    a.kb_per_split = splits > 1 ? kbps : a.num_kb;
    a.num_tiles = a.tiles_m * a.tiles_n * a.splits;
    a.out_rows = static_cast<int>(p->M);
    const bool split = splits > 1;
    // Stream-K: the plan's layout for TMA runs; for class-view runs one laid
    // out here, over their own tiles and k-blocks.
    int sk_tiles = use_tma ? p->sk_tiles : 0, sk_w = use_tma ? p->sk_w : 0;
    if (use_cls && p->choice.sk && !split && p->sk_ctas >= p->slots_cls * k->cg &&
        !sat::sk_layout(tiles_m * tiles_n, a.num_kb, p->slots_cls, &sk_tiles, &sk_w))
        sk_tiles = sk_w = 0;
    const bool sk = sk_tiles > 0;
    const bool pack = (use_tma || use_cls) && !b_rows_ok;
    // Split-K and stream-K runs, and runs whose B must be packed, write this
    // stream's scratch set, held (with the plan's scratch lock)
    // until the run is enqueued and its end recorded.
    std::unique_lock<std::mutex> slock(p->scratch_mu, std::defer_lock);
    Scratch* sc = nullptr;
    if (split || sk || pack) {
        slock.lock();
        const int rc = acquire_scratch(p, stream, pack, &sc);
        if (rc)
            return rc;
    }
    if (split) {
        // The GEMM writes raw fp32 partial tiles to the workspace; the
        // reduction applies alpha and beta.
        a.C = sc->ws;
        a.ldc = static_cast<int>(p->N);
        a.c_half = 0;
        a.alpha = 1.0f;
        a.beta = 0.0f;
        a.out_rows = p->ws_rows;
    }
    a.group = p->choice.group;
    a.raster = p->choice.raster;
    a.alt_k = p->alt_k ? 1 : 0;
    a.err = p->d_err;
    a.timeout_ns = p->timeout_ns;

    // C goes through the bulk-store epilogue when its base and row stride
    // are 16-byte multiples (a TMA store box must start on a 16-byte boundary).
    // (16-bit C always goes through the row-store epilogue.)
    const bool c_tma = split ? sc->ws_tma
                             : p->c_half == 0 && p->N % 4 == 0 && ldc % 4 == 0 &&
                                   reinterpret_cast<uintptr_t>(C) % 16 == 0;
    a.c_tma = c_tma ? 1 : 0;
    a.c_ring = p->c_ring && use_tma && c_tma && !split && beta != 0.0f ? 1 : 0;
    if (sk) {
        // Each launch on a scratch set has its own number; a slot's counter
        // reaches number x (epilogue warps) once its partial tile of this launch
        // is written, and the ticket counter number x slots once every slot of
        // it is handed out. Before the counters could wrap, they are cleared
        // and numbering restarts.
        // A slot's counter counts its partial tiles over the launches on these
        // counters, so every launch must use one layout: a different one (a
        // class-view run after a TMA run, or another alignment of A) clears
        // them first, on the stream, and numbering restarts.
        const unsigned long long sig = (static_cast<unsigned long long>(use_cls ? 1 : 0) << 63) ^
                                       (static_cast<unsigned long long>(sk_tiles) << 32) ^
                                       (static_cast<unsigned long long>(sk_w) << 8) ^
                                       static_cast<unsigned long long>(a.tiles_m);
        unsigned epoch = ++sc->epoch;
        if (epoch >= (1u << 28) || sc->sk_sig != sig) {
            e = cudaMemsetAsync(sc->sk_flags, 0, sk_flag_bytes(p), stream);
            if (e != cudaSuccess)
                return cuda_fail(e, "clearing the stream-K counters");
            sc->epoch = epoch = 1;
            sc->sk_sig = sig;
        }
        a.sk_tiles = sk_tiles;
        a.sk_w = sk_w;
        a.sk_ws = sc->sk_ws;
        a.sk_flags = sc->sk_flags;
        a.sk_ticket = sc->sk_flags + p->sk_ctas + kTicketPad - 1;
        a.sk_epoch = epoch;
    }
    CUtensorMap tmA{}, tmB{}, tmC{};
    if (split && c_tma) {
        tmC = sc->tmW;
    } else if (c_tma) {
        std::lock_guard<std::mutex> lock(p->mu);
        if (p->map_C != C || p->map_ldc != ldc) {
            const int rc =
                encode_2d(&p->tmC, sat::kDtTF32, C, p->N, p->M, 32u, 32u, CU_TENSOR_MAP_SWIZZLE_128B, ldc);
            if (rc) {
                p->map_C = nullptr;
                return rc;
            }
            p->map_C = C;
            p->map_ldc = ldc;
        }
        tmC = p->tmC;
    }
    // B as it lies, or packed into rows of ldb_pack elements (whole 128-byte
    // lines) first, on the same stream.
    const void* bsrc = B;
    int64_t bld = ldb;
    if (pack) {
        e = sat::launch_pack_rows(B, ldb * es64, sc->bpack, p->ldb_pack * es64, p->K, p->N * es64, p->sm_count,
                                  stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "launching the packing of B");
        bsrc = sc->bpack;
        bld = p->ldb_pack;
    }
    if (use_cls) {
        std::lock_guard<std::mutex> lock(p->mu);
        if (p->cls_B != bsrc || p->cls_ldb != bld) {
            const int rc = encode_2d(&p->tmClsB, p->dt, bsrc, p->N, p->K, static_cast<uint32_t>(128 / es),
                                     static_cast<uint32_t>(k->bk), static_cast<CUtensorMapSwizzle>(k->b_swizzle), bld);
            if (rc) {
                p->cls_B = nullptr;
                return rc;
            }
            p->cls_B = bsrc;
            p->cls_ldb = bld;
        }
        tmB = p->tmClsB;
        a.c_tma = 0;
        a.c_ring = 0;
    }
    if (use_tma) {
        std::lock_guard<std::mutex> lock(p->mu);
        // Each operand as it lies: K contiguous (boxes of BK x rows, 128-byte
        // swizzle) or M/N contiguous (boxes of 128 bytes x BK, the MN-major
        // swizzle of the dtype).
        const uint32_t cw = static_cast<uint32_t>(128 / es), bk = static_cast<uint32_t>(k->bk);
        const CUtensorMapSwizzle mn_swz = static_cast<CUtensorMapSwizzle>(k->b_swizzle);
        if (p->map_A != A || p->map_lda != lda) {
            const int rc = p->trans_a ? encode_2d(&p->tmA, p->dt, A, p->M, p->K, cw, bk, mn_swz, lda)
                                      : encode_2d(&p->tmA, p->dt, A, p->K, p->M, bk,
                                                  k->prod == sat::kProdSwap ? static_cast<uint32_t>(k->bn) : 128u,
                                                  CU_TENSOR_MAP_SWIZZLE_128B, lda);
            if (rc) {
                p->map_A = nullptr;
                return rc;
            }
            p->map_A = A;
            p->map_lda = lda;
        }
        if (p->map_B != bsrc || p->map_ldb != bld) {
            const int rc = p->trans_b ? encode_2d(&p->tmB, p->dt, bsrc, p->K, p->N, bk,
                                                  static_cast<uint32_t>(k->bn / k->cg), CU_TENSOR_MAP_SWIZZLE_128B, bld)
                                      : encode_2d(&p->tmB, p->dt, bsrc, p->N, p->K, cw, bk, mn_swz, bld);
            if (rc) {
                p->map_B = nullptr;
                return rc;
            }
            p->map_B = bsrc;
            p->map_ldb = bld;
        }
        tmA = p->tmA;
        tmB = p->tmB;
    }
    if (use_cls) {
        // Class-view tiles write fp32 C rows in 16-byte stores when the rows P
        // apart lie a whole number of 16-byte units apart (unsplit runs
        // without stream-K pieces): rows that start 16-byte aligned always;
        // the others, whose ends take element-wise stores, only where the
        // epilogue is the slower stage, i.e. 16-bit operands (half the MMA
        // time per tile of TF32) with C read as well as written. Measured at
        // (8191, 4097, 2049): bf16 beta 0.5 158 -> 150 us; bf16 beta 0 130 ->
        // 140 us and tf32 beta 0.5 228 -> 240 us, where they are not used.
        if (!split && !sk && p->c_half == 0 && (static_cast<int64_t>(a.a_classes) * ldc) % 4 == 0)
            a.c_cls = p->dt != sat::kDtTF32 && beta != 0.0f ? 2 : 1;
        // Class maps are copied under the lock: another thread may re-encode them.
        CUtensorMap cmaps[sat::kMaxClasses];
        {
            std::lock_guard<std::mutex> lock(p->mu);
            for (int r = 0; r < a.a_classes; ++r)
                cmaps[r] = p->tmCls[r];
        }
        // Every slot runs under stream-K; otherwise one block (pair) per unit, at
        // most the co-resident ones.
        const int64_t units = static_cast<int64_t>(a.num_tiles);
        const int grid =
            static_cast<int>((sk || units >= p->slots_cls ? p->slots_cls : units) * k->cg);
        e = k->launch(cmaps, &tmB, &tmC, &a, grid, stream);
    } else {
        e = k->launch(&tmA, &tmB, &tmC, &a, use_tma ? p->grid_tma : p->grid_plain, stream);
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "launching the GEMM kernel");
    if (split) {
        e = sat::launch_splitk_reduce(sc->ws, splits, static_cast<long long>(p->ws_rows) * p->N, C, p->c_half, p->M,
                                      p->N, ldc, alpha, beta, p->sm_count, stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "launching the split-K reduction");
    }
    if (sc) {
        e = cudaEventRecord(sc->done, stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "recording the end of the run");
    }
    return GEMM_OK;
}

}  // namespace

extern "C" {

gemm_plan* gemm_plan_create(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype)
{
    return create(M, N, K, dtype, nullptr);
}

gemm_plan* gemm_plan_create_config(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, const char* config)
{
    return create(M, N, K, dtype, config);
}

gemm_plan* gemm_plan_create_ex(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, int trans_a, int trans_b,
                               gemm_ctype_t c_type, const char* config)
{
    return create(M, N, K, dtype, config, trans_a != 0, trans_b != 0, static_cast<int>(c_type));
}

void gemm_plan_destroy(gemm_plan* plan)
{
    if (!plan)
        return;
    for (int i = 0; i < plan->n_scratch; ++i)
        free_scratch(plan->scratch[i]);
    for (gemm_plan* sub : plan->host_plan)
        gemm_plan_destroy(sub);
    if (plan->h_err)
        cudaFreeHost(plan->h_err);
    delete plan;
}

const char* gemm_plan_describe(const gemm_plan* plan) { return plan ? plan->desc : ""; }

const char* gemm_last_error(void) { return g_err; }


int gemm_run(const gemm_plan* p, const void* A, const void* B, float* C, float alpha, float beta, void* cuda_stream)
{
    if (!p)
        return fail(GEMM_ERR_ARG, "plan is NULL");
    return run_impl(p, A, p->trans_a ? p->M : p->K, B, p->trans_b ? p->K : p->N, C, p->N, alpha, beta, cuda_stream);
}

int gemm_run_ex(const gemm_plan* p, const void* A, int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                float alpha, float beta, void* cuda_stream)
{
    return run_impl(p, A, lda, B, ldb, C, ldc, alpha, beta, cuda_stream);
}

int gemm_run_host(const gemm_plan* p, const void* hA, const void* hB, float* hC, float alpha, float beta, void* dA,
                  void* dB, float* dC, void* cuda_stream)
{
    if (!p)
        return fail(GEMM_ERR_ARG, "plan is NULL");
    if (p->M == 0 || p->N == 0)
        return GEMM_OK;
    if (!hC || !dC || (p->K > 0 && (!hA || !hB || !dA || !dB)))
        return fail(GEMM_ERR_ARG, "NULL buffer");
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const size_t es = static_cast<size_t>(elem_size(p->dt));
    cudaError_t e = cudaSuccess;
    const size_t cbytes = static_cast<size_t>(p->M * p->N) * sizeof(float);
    // Large untransposed fp32-C problems go in row blocks: B, then each block
    // of A (and of C when beta != 0) copied in on a copy stream, each block's
    // GEMM on `stream` as soon as its rows have arrived, and each block of C
    // copied out on a second copy stream as soon as it is computed. The copies
    // in, the GEMMs and the copies out then overlap.
    const size_t in_bytes = static_cast<size_t>(p->M * p->K + p->K * p->N) * es;
    if (p->K > 0 && alpha != 0.0f && !p->trans_a && !p->trans_b && p->c_half == 0 && p->M >= 1024 &&
        in_bytes >= (size_t(32) << 20)) {
        const int64_t blk = std::max(kHostMinRows, ((p->M + kHostBlocks - 1) / kHostBlocks + 255) / 256 * 256);
        const int nb = static_cast<int>((p->M + blk - 1) / blk);
        const int64_t last = p->M - (nb - 1) * blk;
        gemm_plan* sub[2] = {nullptr, nullptr};
        {
            std::lock_guard<std::mutex> lock(p->mu);
            for (int j = 0; j < 2; ++j) {
                const int64_t rows = j == 0 ? blk : last;
                if (!p->host_plan[j] || p->host_rows[j] != rows) {
                    gemm_plan_destroy(p->host_plan[j]);
                    p->host_plan[j] = create(rows, p->N, p->K, static_cast<gemm_dtype_t>(p->dt), nullptr);
                    p->host_rows[j] = p->host_plan[j] ? rows : 0;
                    if (!p->host_plan[j])
                        return GEMM_ERR_LAUNCH;  // create() set the message
                }
                sub[j] = p->host_plan[j];
            }
        }
        std::lock_guard<std::mutex> slock(p->scratch_mu);
        Scratch* sc = nullptr;
        int rc = acquire_scratch(p, s, false, &sc);
        if (rc)
            return rc;
        if (!sc->cp_in) {
            e = cudaStreamCreateWithFlags(&sc->cp_in, cudaStreamNonBlocking);
            if (e == cudaSuccess)
                e = cudaStreamCreateWithFlags(&sc->cp_out, cudaStreamNonBlocking);
            for (cudaEvent_t& ev : sc->hev)
                if (e == cudaSuccess)
                    e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
            if (e != cudaSuccess)
                return cuda_fail(e, "creating the copy streams of gemm_run_host");
        }
        cudaEvent_t ev_start = sc->hev[0], ev_end = sc->hev[1];
        cudaEvent_t* ev_in = sc->hev + 2;
        cudaEvent_t* ev_done = sc->hev + 2 + kHostBlocks;
        const char* what = "enqueueing gemm_run_host's row blocks";
        // Copies in wait for everything before this call on `stream`.
        e = cudaEventRecord(ev_start, s);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(sc->cp_in, ev_start, 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dB, hB, static_cast<size_t>(p->K * p->N) * es, cudaMemcpyHostToDevice, sc->cp_in);
        for (int b = 0; b < nb && e == cudaSuccess; ++b) {
            const int64_t r0 = b * blk, rows = b == nb - 1 ? last : blk;
            e = cudaMemcpyAsync(static_cast<char*>(dA) + r0 * p->K * es, static_cast<const char*>(hA) + r0 * p->K * es,
                                static_cast<size_t>(rows * p->K) * es, cudaMemcpyHostToDevice, sc->cp_in);
            if (e == cudaSuccess && beta != 0.0f)
                e = cudaMemcpyAsync(dC + r0 * p->N, hC + r0 * p->N, static_cast<size_t>(rows * p->N) * sizeof(float),
                                    cudaMemcpyHostToDevice, sc->cp_in);
            if (e == cudaSuccess)
                e = cudaEventRecord(ev_in[b], sc->cp_in);
        }
        if (e != cudaSuccess)
            return cuda_fail(e, what);
        for (int b = 0; b < nb; ++b) {
            const int64_t r0 = b * blk;
            e = cudaStreamWaitEvent(s, ev_in[b], 0);
            if (e != cudaSuccess)
                return cuda_fail(e, what);
            rc = gemm_run(sub[b == nb - 1 ? 1 : 0], static_cast<const char*>(dA) + r0 * p->K * es, dB, dC + r0 * p->N,
                          alpha, beta, cuda_stream);
            if (rc)
                return rc;
            e = cudaEventRecord(ev_done[b], s);
            if (e == cudaSuccess)
                e = cudaStreamWaitEvent(sc->cp_out, ev_done[b], 0);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(hC + r0 * p->N, dC + r0 * p->N,
                                    static_cast<size_t>((b == nb - 1 ? last : blk) * p->N) * sizeof(float),
                                    cudaMemcpyDeviceToHost, sc->cp_out);
            if (e != cudaSuccess)
                return cuda_fail(e, what);
        }
        // `stream` continues once the last block of C is on the host.
        e = cudaEventRecord(ev_end, sc->cp_out);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(s, ev_end, 0);
        if (e == cudaSuccess)
            e = cudaEventRecord(sc->done, s);
        return e == cudaSuccess ? GEMM_OK : cuda_fail(e, what);
    }
    if (p->K > 0 && alpha != 0.0f) {
        e = cudaMemcpyAsync(dA, hA, static_cast<size_t>(p->M * p->K) * es, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dB, hB, static_cast<size_t>(p->K * p->N) * es, cudaMemcpyHostToDevice, s);
    }
    if (e == cudaSuccess && beta != 0.0f)
        e = cudaMemcpyAsync(dC, hC, cbytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "copying operands to the device");
    const int rc = gemm_run(p, dA, dB, dC, alpha, beta, cuda_stream);
    if (rc)
        return rc;
    e = cudaMemcpyAsync(hC, dC, cbytes, cudaMemcpyDeviceToHost, s);
    return e == cudaSuccess ? GEMM_OK : cuda_fail(e, "copying C to the host");
}

int gemm_plan_status(const gemm_plan* p)
{
    if (!p)
        return fail(GEMM_ERR_ARG, "plan is NULL");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return cuda_fail(e, "device error");
    volatile uint32_t* w = reinterpret_cast<volatile uint32_t*>(p->h_err);
    uint32_t h = *w;
    *w = 0;
    for (const gemm_plan* sub : p->host_plan)
        if (sub && gemm_plan_status(sub) == GEMM_ERR_TIMEOUT)
            h |= 1u << 31;  // a row block of gemm_run_host gave up a wait
    if (h) {
        // A launch that gave up may have left stream-K counters short of its
        // number: start the numbering again from cleared counters.
        std::lock_guard<std::mutex> lock(p->scratch_mu);
        for (int i = 0; i < p->n_scratch; ++i) {
            Scratch& s = p->scratch[i];
            if (s.sk_flags && cudaMemset(s.sk_flags, 0, sk_flag_bytes(p)) == cudaSuccess)
                s.epoch = 0;
        }
        return fail(GEMM_ERR_TIMEOUT, "a bounded wait gave up inside the kernel (error bits 0x%x)", h);
    }
    return GEMM_OK;
}

int gemm_selftest_bounded_wait(uint64_t timeout_ns)
{
    if (timeout_ns > 1000000000ull)
        timeout_ns = 1000000000ull;
    uint32_t* d = nullptr;
    cudaError_t e = cudaMalloc(&d, sizeof(uint32_t));
    if (e == cudaSuccess)
        e = cudaMemset(d, 0, sizeof(uint32_t));
    if (e == cudaSuccess)
        e = sat::launch_wait_probe(d, timeout_ns, nullptr);
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    uint32_t h = 0;
    if (e == cudaSuccess)
        e = cudaMemcpy(&h, d, sizeof h, cudaMemcpyDeviceToHost);
    if (d)
        cudaFree(d);
    if (e != cudaSuccess)
        return cuda_fail(e, "bounded-wait self-test");
    if (h & (1u << 4))
        return fail(GEMM_ERR_TIMEOUT, "the probe's wait gave up after its limit, as designed");
    return fail(GEMM_ERR_LAUNCH, "the probe's wait did not report a timeout (error word 0x%x)", h);
}

int gemm_select_config(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, int sm_count, int tma_ok, char* out,
                       int out_len)
{
    const int dt = static_cast<int>(dtype);
    if (M < 0 || N < 0 || K < 0 || dt < 0 || dt > 2 || sm_count < 1 || !out || out_len < 1)
        return fail(GEMM_ERR_ARG, "bad arguments to gemm_select_config");
    const sat::Choice c = sat::select_config(M, N, K, dt, sm_count, tma_ok != 0);
    // The ring depth of the kernel the choice names (the plain-load kernel's
    // when TMA cannot read the operands).
    const sat::KernelEntry* k = tma_ok ? sat::find_entry(dt, c.bn, c.cg, c.swap ? sat::kProdSwap : sat::kProdTMA,
                                                         c.swap ? 0 : c.stages)
                                       : sat::find_entry(dt, c.cg == 2 ? 256 : (c.bn < 128 ? 128 : c.bn), c.cg,
                                                         sat::kProdClassA);
    std::snprintf(out, static_cast<size_t>(out_len), "%d,%d,%d,%d,%d,%d,%d,%d,%d,%s", c.bn, c.cg, c.raster, c.group,
                  c.splits > 1 ? c.splits : 1, c.cload, c.sk, c.swap, k ? k->stages : 0,
                  c.source == sat::kSrcTable ? "table" : c.source == sat::kSrcBucket ? "bucket" : "rule");
    return GEMM_OK;
}

}  // extern "C"
