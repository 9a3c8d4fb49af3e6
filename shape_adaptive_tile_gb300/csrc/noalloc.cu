// gemm_run_noalloc: the GEMM for callers that must not allocate memory.
//
// Some callers cannot call cudaMalloc or cudaFree once they are running. A
// framework may have reserved the device's memory for its own pool, cudaFree
// synchronises the device (which a latency-bound loop cannot afford), and some
// host programs forbid device allocation after start-up. gemm_plan_create
// allocates (host state, an error word and, for split-K plans, a workspace),
// so such callers use this entry point instead. It needs no plan: the
// dispatcher's choice, the tensor maps and the launch parameters live on the
// stack, and the kernel's scratch memory (its status word, the stream-K
// counters, and the split-K or stream-K partial tiles) lives in one
// file-scope device array of fixed size that every GPU loading this library
// holds until the process exits.
#include "gemm.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "dispatch.h"
#include "registry.h"

namespace {

// 32 MiB: 4 KiB for the status word (offset 0), the stream-K slot ticket
// (offset 128) and the stream-K counters (offset 256, one per CTA), the rest
// for split-K or stream-K partial tiles.
constexpr size_t kScratchBytes = size_t(32) << 20;
constexpr size_t kStatusBytes = 4096;
constexpr size_t kTicketOffset = 128;
constexpr size_t kCounterOffset = 256;
constexpr size_t kWorkspaceBytes = kScratchBytes - kStatusBytes;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    void* scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int sm_count = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Row-major 2-D tensor map, 128-byte-swizzled boxes, zero fill outside.
bool encode(CUtensorMap* map, CUtensorMapDataType t, int es, const void* ptr, uint64_t inner, uint64_t outer,
            uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz)
{
    return sat::encode_map(map, t, es, ptr, inner, outer, inner, box_inner, box_outer, swz) == 0;
}

// First call on a device, with that device current: look up where the
// scratch array lives on it. Later calls reuse the address.
int setup_device(int dev, DeviceState** out)
{
    if (dev < 0 || dev >= kMaxDevices)
        return sat::fail_with(GEMM_ERR_ARG, "device %d is beyond the %d devices this entry point tracks", dev,
                              kMaxDevices);
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& s = g_dev[dev];
    if (!s.ready) {
        int major = 0, minor = 0, sms = 0;
        cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return sat::fail_with(GEMM_ERR_LAUNCH, "querying device %d: %s", dev, cudaGetErrorString(e));
        if (major != 10 || minor != 3)
            return sat::fail_with(GEMM_ERR_ARCH,
                                  "device %d is compute capability %d.%d; this library is built for sm_103a only",
                        dev, major, minor);
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr)
            return sat::fail_with(GEMM_ERR_LAUNCH, "cudaGetSymbolAddress of the scratch array on device %d: %s", dev,
                        cudaGetErrorString(e));
        s.scratch = ptr;
        s.sm_count = sms;
        s.ready = true;
    }
    *out = &s;
    return GEMM_OK;
}

// CTA slots (single CTAs, or pairs) that can be resident at once.
int64_t slots_for(int sm_count, const sat::KernelEntry* e)
{
    int64_t slots = sm_count / e->cg;
    if (e->cg == 2) {
        const int n = e->max_clusters();
        if (n > 0 && n < slots)
            slots = n;
    }
    return slots < 1 ? 1 : slots;
}

int grid_for(int64_t M, int64_t N, int splits, int sm_count, const sat::KernelEntry* e)
{
    int64_t tm = 0, tn = 0;
    sat::tile_grid(e, M, N, &tm, &tn);
    const int64_t units = tm * tn * splits;
    const int64_t slots = slots_for(sm_count, e);
    return static_cast<int>((units < slots ? units : slots) * e->cg);
}

}  // namespace

extern "C" int gemm_run_noalloc(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, const void* A, const void* B,
                                float* C, float alpha, float beta, void* cuda_stream)
{
    sat::set_last_error("");
    const int dt = static_cast<int>(dtype);
    if (M < 0 || N < 0 || K < 0 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
        return sat::fail_with(GEMM_ERR_ARG, "dimensions must be in [0, 2^31)");
    if (dt < 0 || dt > 2)
        return sat::fail_with(GEMM_ERR_ARG, "unknown dtype %d", dt);
    if (M == 0 || N == 0)
        return GEMM_OK;
    if (!C)
        return sat::fail_with(GEMM_ERR_ARG, "C is NULL");
    if (reinterpret_cast<uintptr_t>(C) % 4 != 0)
        return sat::fail_with(GEMM_ERR_ALIGN, "C must be 4-byte aligned");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return sat::fail_with(GEMM_ERR_LAUNCH, "cudaGetDevice: %s", cudaGetErrorString(e));
    DeviceState* ds = nullptr;
    int rc = setup_device(dev, &ds);
    if (rc)
        return rc;
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    if (K == 0 || alpha == 0.0f) {
        e = sat::launch_scale(C, 0, M, N, N, beta, stream);
        return e == cudaSuccess ? GEMM_OK
                                : sat::fail_with(GEMM_ERR_LAUNCH, "beta-scale kernel: %s", cudaGetErrorString(e));
    }
    if (!A || !B)
        return sat::fail_with(GEMM_ERR_ARG, "A or B is NULL");
    const int es = dt == 0 ? 4 : 2;
    if (reinterpret_cast<uintptr_t>(A) % es || reinterpret_cast<uintptr_t>(B) % es)
        return sat::fail_with(GEMM_ERR_ALIGN, "A and B must be aligned to their %d-byte element size", es);

    // The same choice gemm_plan_create would make.
    const bool tma_ok = (K * es) % 16 == 0 && (N * es) % 16 == 0;
    const sat::Choice c = sat::select_config(M, N, K, dt, ds->sm_count, tma_ok);
    const bool use_tma = tma_ok && reinterpret_cast<uintptr_t>(A) % 16 == 0 && reinterpret_cast<uintptr_t>(B) % 16 == 0;
    const sat::KernelEntry* k = use_tma ? sat::find_entry(dt, c.bn, c.cg, c.swap ? sat::kProdSwap : sat::kProdTMA,
                                                          c.swap ? 0 : c.stages)
                                        : sat::find_entry(dt, c.bn < 128 ? 128 : c.bn, 1, sat::kProdPlain);
    if (!k)
        return sat::fail_with(GEMM_ERR_ARG, "no compiled kernel for the chosen configuration");
    const int64_t num_kb = (K + k->bk - 1) / k->bk;
    int splits = c.splits > 1 && num_kb > 1 ? c.splits : 1;
    if (splits > num_kb)
        splits = static_cast<int>(num_kb);
    const int kbps = static_cast<int>((num_kb + splits - 1) / splits);
    if (splits > 1)
        splits = static_cast<int>((num_kb + kbps - 1) / kbps);
    const int64_t tile_rows = 128 * k->cg;  // slices padded to whole tiles only
    const int64_t ws_rows = (M + tile_rows - 1) / tile_rows * tile_rows;
    const size_t ws_bytes = splits > 1 ? static_cast<size_t>(splits) * ws_rows * static_cast<size_t>(N) * 4 : 0;
    if (ws_bytes > kWorkspaceBytes)
        return sat::fail_with(GEMM_ERR_ARG,
                    "this problem splits K %d ways and needs %zu bytes of scratch; the allocation-free entry point "
                    "has %zu bytes (use gemm_plan_create/gemm_run, which allocate their own workspace)",
                    splits, ws_bytes, kWorkspaceBytes);
    // Stream-K, laid out as gemm_plan_create lays it out.
    int sk_tiles = 0, sk_w = 0;
    int64_t sk_ctas = 0;
    if (c.sk && use_tma && splits == 1) {
        int64_t tm = 0, tn = 0;
        sat::tile_grid(k, M, N, &tm, &tn);
        const int64_t tiles = tm * tn;
        const int64_t slots = slots_for(ds->sm_count, k);
        if (sat::sk_layout(tiles, num_kb, slots, &sk_tiles, &sk_w)) {
            sk_ctas = slots * k->cg;
            const size_t need = static_cast<size_t>(sk_ctas) * 128 * k->bn * 4;
            if (need > kWorkspaceBytes)
                return sat::fail_with(GEMM_ERR_ARG,
                            "this problem's stream-K partial tiles need %zu bytes of scratch; the allocation-free "
                            "entry point has %zu bytes (use gemm_plan_create/gemm_run)",
                            need, kWorkspaceBytes);
            if (kCounterOffset + static_cast<size_t>(sk_ctas) * 4 > kStatusBytes)
                return sat::fail_with(GEMM_ERR_ARG,
                            "this problem's stream-K grid has %lld CTAs, each needing a counter; the "
                            "allocation-free entry point has %zu counter slots (use gemm_plan_create/gemm_run)",
                            static_cast<long long>(sk_ctas), (kStatusBytes - kCounterOffset) / 4);
        }
    }
    e = k->prepare();
    if (e != cudaSuccess)
        return sat::fail_with(GEMM_ERR_LAUNCH, "setting the kernel's shared-memory limit: %s", cudaGetErrorString(e));

    uint32_t* status = static_cast<uint32_t*>(ds->scratch);
    float* ws = reinterpret_cast<float*>(static_cast<unsigned char*>(ds->scratch) + kStatusBytes);
    // The array keeps the previous call's contents; the status word, the
    // stream-K ticket and counters must start at zero (this call is launch
    // number 1).
    e = cudaMemsetAsync(status, 0, kStatusBytes, stream);
    if (e != cudaSuccess)
        return sat::fail_with(GEMM_ERR_LAUNCH, "clearing the status word: %s", cudaGetErrorString(e));

    sat::GemmArgs a{};
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.A = A;
    a.B = B;
    a.lda = static_cast<int>(K);
    a.ldb = static_cast<int>(N);
    a.ldc = static_cast<int>(N);
    a.C = splits > 1 ? ws : C;
    a.alpha = splits > 1 ? 1.0f : alpha;
    a.beta = splits > 1 ? 0.0f : beta;
    int64_t tiles_m = 0, tiles_n = 0;
    sat::tile_grid(k, M, N, &tiles_m, &tiles_n);
    a.tiles_m = static_cast<int>(tiles_m);
    a.tiles_n = static_cast<int>(tiles_n);
    a.num_kb = static_cast<int>(num_kb);
    a.splits = splits;
    a.kb_per_split = splits > 1 ? kbps : a.num_kb;
    a.num_tiles = a.tiles_m * a.tiles_n * splits;
    a.out_rows = splits > 1 ? static_cast<int>(ws_rows) : static_cast<int>(M);
    a.group = c.group;
    a.raster = c.raster;
    a.alt_k = 1;
    a.err = status;
    a.timeout_ns = 2000000000ull;

    const CUtensorMapDataType tdt = dt == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                    : dt == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tmA{}, tmB{}, tmC{};
    const bool c_tma = (N * 4) % 16 == 0 && (splits > 1 || reinterpret_cast<uintptr_t>(C) % 16 == 0);
    if (c_tma && !encode(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.C, N,
                         splits > 1 ? static_cast<uint64_t>(splits) * ws_rows : static_cast<uint64_t>(M), 32u, 32u,
                         CU_TENSOR_MAP_SWIZZLE_128B))
        return sat::fail_with(GEMM_ERR_LAUNCH, "encoding the output tensor map");
    a.c_tma = c_tma ? 1 : 0;
    a.c_ring = !c.cload && use_tma && k->c_ring && c_tma && splits == 1 && sk_tiles == 0 && beta != 0.0f ? 1 : 0;
    if (sk_tiles > 0) {
        a.sk_tiles = sk_tiles;
        a.sk_w = sk_w;
        a.sk_ws = ws;
        a.sk_flags = reinterpret_cast<unsigned*>(static_cast<unsigned char*>(ds->scratch) + kCounterOffset);
        a.sk_ticket = reinterpret_cast<unsigned*>(static_cast<unsigned char*>(ds->scratch) + kTicketOffset);
        a.sk_epoch = 1;
    }
    if (use_tma) {
        if (!encode(&tmA, tdt, es, A, K, M, static_cast<uint32_t>(k->bk),
                    k->prod == sat::kProdSwap ? static_cast<uint32_t>(k->bn) : 128u, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode(&tmB, tdt, es, B, N, K, static_cast<uint32_t>(128 / es), static_cast<uint32_t>(k->bk),
                    static_cast<CUtensorMapSwizzle>(k->b_swizzle)))
            return sat::fail_with(GEMM_ERR_LAUNCH, "encoding the operand tensor maps");
    }
    const int grid = sk_tiles > 0 ? static_cast<int>(sk_ctas) : grid_for(M, N, splits, ds->sm_count, k);
    e = k->launch(&tmA, &tmB, &tmC, &a, grid, stream);
    if (e != cudaSuccess)
        return sat::fail_with(GEMM_ERR_LAUNCH, "launching the GEMM kernel: %s", cudaGetErrorString(e));
    if (splits > 1) {
        e = sat::launch_splitk_reduce(ws, splits, static_cast<long long>(ws_rows) * N, C, 0, M, N, N, alpha, beta,
                                      ds->sm_count, stream);
        if (e != cudaSuccess)
            return sat::fail_with(GEMM_ERR_LAUNCH, "launching the split-K reduction: %s", cudaGetErrorString(e));
    }
    return GEMM_OK;
}
