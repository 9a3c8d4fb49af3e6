/*
 * Deterministic, shape-adaptive dense GEMM for GB300 (sm_103a): the C ABI.
 *
 *     C = alpha * A * B + beta * C
 *
 * A is M x K, B is K x N, C is M x N, all dense row-major with no padding
 * (lda = K, ldb = N, ldc = N) and no transposes. A and B are fp32 (computed
 * on the TF32 tensor cores), bf16 or fp16; accumulation and C are fp32.
 *
 * The operation is the GEMM that "Scale coverage exposes a remaining GEMM
 * gap" measures (section "Measurement contract and evidence": C = A*B,
 * alpha = 1, beta = 0, compact row-major, no transpose) in its BLAS form
 * with alpha and beta. "Measured data point on fixed-tile vs shape-adaptive
 * GEMM" (section "The wall, and why we think it's structural") argues that
 * what such a library must provide is a per-shape choice of tile and
 * schedule, not one kernel; gemm_plan_create makes that choice once per
 * (M, N, K, dtype), and gemm_run executes it. Its section "The actual
 * question" names the constraint kept here: results are bit-identical from
 * run to run (no split-K with atomics, a fixed K order per output tile).
 *
 * All device pointers are plain CUDA device addresses (for example
 * torch.Tensor.data_ptr()); the library never allocates, frees or keeps
 * them. Functions return 0 on success or a negative gemm_status_t; the
 * message of the last failure on the calling thread is in gemm_last_error().
 */
#ifndef SAT_GEMM_H
#define SAT_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of A and B. C is always fp32. */
typedef enum {
    GEMM_TF32 = 0, /* fp32 storage, TF32 tensor-core multiply, fp32 accumulate */
    GEMM_BF16 = 1, /* bfloat16 storage, fp32 accumulate */
    GEMM_FP16 = 2  /* IEEE binary16 storage, fp32 accumulate */
} gemm_dtype_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_ARG = -1,     /* NULL plan/pointer, negative or oversized dimension, bad dtype */
    GEMM_ERR_ARCH = -2,    /* current device is not compute capability 10.3 (sm_103) */
    GEMM_ERR_ALIGN = -3,   /* A/B not aligned to their element size, or C not 4-byte aligned */
    GEMM_ERR_LAUNCH = -4,  /* a CUDA call failed (message in gemm_last_error) */
    GEMM_ERR_TIMEOUT = -5, /* a bounded wait inside a kernel gave up (see gemm_plan_status) */
    GEMM_ERR_NOMEM = -6    /* host or device allocation failed while creating a plan */
} gemm_status_t;

typedef struct gemm_plan gemm_plan; /* opaque */

/* Element type of C for gemm_plan_create_ex (accumulation is fp32 either way). */
typedef enum {
    GEMM_C_F32 = 0,  /* fp32 */
    GEMM_C_BF16 = 1, /* bfloat16, rounded to nearest even */
    GEMM_C_F16 = 2   /* IEEE binary16, rounded to nearest even */
} gemm_ctype_t;

/*
 * Choose the kernel (tile shape, CTA-pair or single SM, stage count, raster
 * order, load path) for this problem on the CURRENT device, and prepare it.
 * M, N, K >= 0 and each < 2^31. Allocates host state and a 64-byte
 * host-mapped pinned error word, both owned by the plan. A plan whose choice
 * splits K, or cuts the last waves of tiles into stream-K pieces, also owns
 * device scratch for its partial tiles, one set per stream it runs on (at
 * most 8 sets), allocated by the first run on each stream: a split-K set is
 * splits x ceil(M/256)*256 x N floats; a stream-K set one 128 x bn float
 * partial tile and one counter per CTA of the grid (at most one per SM),
 * plus a slot ticket. Returns NULL on failure; the reason is in
 * gemm_last_error(). Must not be called during CUDA stream capture.
 */
gemm_plan* gemm_plan_create(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype);

/*
 * As gemm_plan_create, but with the dispatcher's choice replaced by
 * `config` = "bn,cg,raster,group[,splits]" (bn in {64,128,256}; cg 1 or 2,
 * where 2 needs bn >= 128; raster 0 = groups along M, 1 = along N;
 * group >= 1; splits 1..16 K splits, default 1), optionally followed by
 * ",st<n>" (a ring of n shared-memory stages where the untransposed TMA
 * kernel of that tile is compiled with that depth; the deepest by default),
 * ",fwd" (every wave of tiles runs through K forwards; by default alternate
 * waves run it backwards, starting on the operand panels the previous wave
 * left in L2; either order is fixed per tile, so results repeat bit for bit),
 * ",cload" (with beta != 0 the epilogue loads C itself instead of the
 * producer fetching it through the operand ring), ",swap" (operand roles
 * exchanged: the tensor core computes C^T = B^T A^T in tiles of 128 columns
 * by bn rows of C; cg 1, bn 64 or 128), ",sk" (stream-K: the
 * tiles of the last full wave and the partial one are cut into equal
 * k-block ranges, one per CTA slot, and each split tile's pieces are added
 * in fixed order) and ",plain" (force the plain-load producer). NULL or ""
 * means the dispatcher decides. For sweeps and tests; every configuration
 * computes the same GEMM (with splits > 1 or stream-K the K sum of some
 * tiles is cut into fixed slices whose partial sums are added in fixed
 * order, so the bits can differ from the unsplit order but are identical
 * from run to run).
 */
gemm_plan* gemm_plan_create_config(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, const char* config);

/*
 * As gemm_plan_create_config, for C = alpha * op(A) * op(B) + beta * C where
 * op(A) is M x K and op(B) is K x N: trans_a != 0 means A is stored as its
 * transpose (K x M, row-major), trans_b != 0 that B is (N x K, row-major).
 * c_type gives C's element type: with GEMM_C_BF16 or GEMM_C_F16 the
 * epilogue reads C (beta != 0) and writes it in that type, computing
 * alpha * acc + beta * C in fp32 and rounding once to nearest even; such C
 * is written row by row (no bulk-store epilogue, no C through the ring).
 * Transposed operands are read by TMA only (no plain-load kernel exists for
 * them), so every gemm_run_ex of such a plan needs A and B 16-byte aligned
 * with row strides that are multiples of 16 bytes (GEMM_ERR_ALIGN
 * otherwise). Tiles with transposed operands are 1-SM 128 x 128 or
 * 128 x 256, or CTA-pair 256 x 256; a configuration naming another tile N
 * is rounded to one of these, and ",swap" is ignored. `config` may be NULL.
 */
gemm_plan* gemm_plan_create_ex(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, int trans_a, int trans_b,
                               gemm_ctype_t c_type, const char* config);

/*
 * Enqueue C = alpha * A * B + beta * C on `cuda_stream` (a cudaStream_t; NULL
 * is the legacy default stream) and return without synchronising.
 *   A: device pointer, M x K elements of the plan's dtype, row-major.
 *   B: device pointer, K x N elements, row-major.
 *   C: device pointer, M x N floats, row-major; read only if beta != 0
 *      (so with beta == 0 any contents, NaN included, are ignored).
 * M == 0 or N == 0: nothing is done. K == 0 or alpha == 0: C = beta * C.
 * A and B must be aligned to their element size, C to 4 bytes
 * (GEMM_ERR_ALIGN otherwise). Rows that TMA can address (16-byte aligned
 * starts) are read as they lie. Otherwise (untransposed plans): A is read
 * through one tensor map per residue class of its row starts modulo 16
 * bytes, and B is first copied, by a kernel on the same stream, into rows of
 * whole 128-byte lines in scratch of the stream's own (allocated by the
 * plan's first such run on that stream). Every path sums K in a fixed
 * order; the class views start their k-blocks a few elements earlier, so
 * their results can differ from the aligned path's by rounding (and are
 * identical where every partial sum is exact). A plan that splits K launches
 * a second kernel on the same stream that sums the partial tiles in fixed
 * order and applies alpha and beta.
 * Threading: one plan may run on several streams, from several threads, at
 * once. A split-K or stream-K plan keeps its partial tiles in scratch of the
 * stream's own (allocated by the plan's first run on that stream, so make
 * that first run before any stream capture; past 8 streams, a new stream
 * takes over the set used least recently, ordered behind that set's last
 * run by an event wait on the GPU). Stream-K CTAs wait for partial tiles
 * only of CTAs that started before them (slots are handed out in start
 * order), so such runs finish whether or not the whole grid is resident,
 * beside each other or beside other work.
 * Errors: launch failures return GEMM_ERR_LAUNCH. A kernel of this plan that
 * gave up a bounded wait marks the plan's host-mapped error word; the next
 * gemm_run of the plan sees it without synchronising and returns
 * GEMM_ERR_TIMEOUT with nothing enqueued, until gemm_plan_status() clears it.
 */
int gemm_run(const gemm_plan* plan, const void* A, const void* B, float* C, float alpha, float beta,
             void* cuda_stream);

/*
 * gemm_run with row strides (leading dimensions, in elements): lda for A as
 * stored (>= K, or >= M when the plan has A transposed), ldb for B as stored
 * (>= N, or >= K when transposed), ldc for C (>= N, in elements of the
 * plan's C type; C points to elements of that type, aligned to their size).
 * gemm_run is this call with the dense strides. Operand rows that TMA cannot
 * address (strides that are not 16-byte multiples) take the class views of A
 * and the packed copy of B described at gemm_run (untransposed plans only;
 * a transposed plan returns GEMM_ERR_ALIGN for them); C whose base or row
 * stride is not a 16-byte multiple takes the row-store epilogue.
 * GEMM_ERR_ARG for a stride below the minimum.
 */
int gemm_run_ex(const gemm_plan* plan, const void* A, int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                float alpha, float beta, void* cuda_stream);

/*
 * End-to-end form of gemm_run for operands in HOST memory (pinned host
 * memory gives asynchronous copies): copy hA -> dA, hB -> dB and (only if
 * beta != 0) hC -> dC, run the GEMM on the device buffers, then copy
 * dC -> hC, all ordered on `cuda_stream` (after its earlier work, before its
 * later work). dA, dB, dC are caller-owned device buffers of the full
 * operand sizes. Large untransposed plans with fp32 C (M >= 1024 and at least
 * 32 MiB of A and B) run in up to 8 row blocks of 512 rows or more, whose
 * copies overlap the GEMMs: the copies go on two streams of the calling
 * stream's own (made by
 * the plan's first such run on it), the blocks' GEMMs on `cuda_stream`
 * through plans of the block's shape (made by the first such run and kept
 * with the plan; gemm_plan_status reports their bounded-wait timeouts too).
 * Returns after enqueueing; synchronise the stream before reading hC.
 */
int gemm_run_host(const gemm_plan* plan, const void* hA, const void* hB, float* hC, float alpha, float beta,
                  void* dA, void* dB, float* dC, void* cuda_stream);

/*
 * Allocation-free GEMM. The pages have no counterpart to this entry point; it
 * exists for callers that must not allocate device or host memory while they
 * run: a framework that has reserved the device memory for its own pool, a
 * latency-bound loop that cannot afford cudaFree's device synchronisation,
 * or a host program that forbids device allocation after start-up.
 * gemm_plan_create allocates (host state, an error word, a split-K
 * workspace), so such callers use this instead.
 *
 * Computes the same C = alpha * A * B + beta * C as gemm_run, with the same
 * arguments, conventions, alignment rules and the dispatcher's choice of
 * kernel, but makes no plan and calls no cudaMalloc, cudaFree or other
 * allocating routine. The kernel's scratch memory is one fixed 32 MiB
 * device array inside the library, which every GPU that loads the library
 * holds until the process exits. Its first 4 KiB hold the status word
 * (offset 0), the stream-K slot ticket (offset 128) and the stream-K
 * counters (from offset 256: at most 960, one per CTA of the grid); the
 * other 32 MiB - 4 KiB hold the split-K partial
 * tiles (splits x M rounded up to the tile height, 128 or 256 rows, x N
 * floats) or the stream-K partial tiles (one 128 x bn float tile per CTA).
 *   - A problem whose partial tiles or counters would not fit is rejected
 *     with GEMM_ERR_ARG and a message naming the limit; gemm_run serves it.
 *     On a 152-SM GB300 no choice of the dispatcher comes near either limit
 *     (its K splits and stream-K grids keep the partial tiles within one
 *     128 x 256 float tile per SM, 19.9 MB), so the check guards devices
 *     with more SMs.
 *   - The first call on each device looks up the array's address on that
 *     device (so the device must be current); make that first call before
 *     any CUDA stream capture.
 *   - Every call shares the array, which keeps the previous call's contents;
 *     the status word, the ticket and the counters are cleared on the stream at the
 *     start of each call. Calls whose kernels overlap on the GPU (different
 *     streams, or the same stream from several threads without ordering)
 *     race on the array and may produce wrong results: order them.
 *   - A bounded wait that gives up inside the kernel still ends it; this
 *     entry point has no status query (plans have gemm_plan_status).
 * Returns 0 after enqueueing on `cuda_stream`, or a negative gemm_status_t
 * with the reason in gemm_last_error().
 */
int gemm_run_noalloc(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, const void* A, const void* B, float* C,
                     float alpha, float beta, void* cuda_stream);

/* Free the plan, its error word and its scratch. NULL is accepted.
 * Synchronises nothing: do not destroy a plan whose runs may still be
 * executing. */
void gemm_plan_destroy(gemm_plan* plan);

/*
 * Synchronise the device, read and clear the plan's error word (and, if it
 * was set, clear the stream-K counters of every scratch set, whose numbering
 * a launch that gave up may have left short).
 * Returns 0 if no kernel of this plan gave up a bounded wait since the last
 * call, GEMM_ERR_TIMEOUT if one did, GEMM_ERR_LAUNCH if the device reported
 * an error.
 */
int gemm_plan_status(const gemm_plan* plan);

/* Human-readable description of the chosen configuration, valid for the
 * plan's lifetime, e.g. "tf32 m2048 n2048 k2048: bn256 cg1 st4 tma raster0 g8 grid128". */
const char* gemm_plan_describe(const gemm_plan* plan);

/* Message of the last failure on the calling thread ("" if none). */
const char* gemm_last_error(void);

/*
 * Self-test of the kernels' bounded waits: launch one CTA that waits on a
 * shared-memory barrier nobody arrives at, with a limit of `timeout_ns`
 * (capped at 1 s), then read the error word. Returns GEMM_ERR_TIMEOUT when
 * the wait gave up as designed and the context is still usable, another
 * negative status otherwise. Blocks until the kernel has finished.
 */
int gemm_selftest_bounded_wait(uint64_t timeout_ns);

/*
 * Prepare the device-routine form of the GEMM (include/gemm_device.cuh) for
 * C = alpha * A * B + beta * C on the CURRENT device: writes a
 * gemm_device_params (tensor maps of A, B and C, the persistent schedule,
 * and the launch shape: threads, dynamic shared memory, cluster size, grid)
 * into `params` (host memory, at least `params_bytes` bytes, 64-byte
 * aligned). cta_group 1 selects the 1-SM 128 x 128 tile, 2 the CTA-pair
 * 256 x 256 tile. Dense row-major operands in device memory, 16-byte aligned,
 * with row strides that are multiples of 16 bytes and N a multiple of 4
 * (GEMM_ERR_ALIGN otherwise). The params hold device pointers only; nothing
 * is allocated. The routine has no error word: a bounded wait that gives up
 * shows only in the result. Returns 0 or a negative gemm_status_t.
 */
int gemm_device_prepare(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, const void* A, const void* B, float* C,
                        float alpha, float beta, int cta_group, void* params, int64_t params_bytes);

/*
 * The device routine inside a kernel of the library's own: a persistent
 * kernel prepared by gemm_device_prepare() whose phase 1 is
 * gemm_device_run (C = alpha * A * B + beta * C) and whose phase 2, in the
 * same launch, replaces each element of the tiles the CTA produced by
 * max(x, 0). cta_group as for gemm_device_prepare (1: 128 x 128 tiles,
 * 2: CTA pairs, 256 x 256). For tests: it shows that the routine composes
 * with other work in one launch, for either tile.
 */
int gemm_selftest_device_call(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, const void* A, const void* B,
                              float* C, float alpha, float beta, int cta_group, void* cuda_stream);

/*
 * Host-only view of the dispatcher (no device is touched): the choice that
 * gemm_plan_create would make for this problem on a device with `sm_count`
 * SMs, given whether the TMA path is possible (`tma_ok`: K and N row
 * strides are multiples of 16 bytes). Writes
 * "bn,cg,raster,group,splits,cload,sk,swap,stages,source" (cload: 1 if,
 * with beta != 0, the epilogue loads C itself, 0 if the producer fetches it
 * through the operand ring where the kernel allows; sk: 1 for a stream-K
 * schedule of the last waves; swap: 1 if the tensor core computes C^T =
 * B^T A^T, with bn rows of C per tile; stages: the shared-memory ring depth
 * of the chosen kernel; source: table for an exact hit in the committed
 * sweep table, bucket for the nearest table shape in the same power-of-two
 * bucket of M, N and K, rule for the analytic rule) into `out`
 * (NUL-terminated, at most `out_len` bytes). Returns 0, or GEMM_ERR_ARG on
 * bad arguments.
 */
int gemm_select_config(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, int sm_count, int tma_ok, char* out,
                       int out_len);

#ifdef __cplusplus
}
#endif

#endif /* SAT_GEMM_H */
