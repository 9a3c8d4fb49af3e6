// Small kernels around the GEMM: C = beta * C for K == 0 or alpha == 0, row
// packing of operands whose rows are not 16-byte aligned, the split-K
// reduction, the registry lookup, and the bounded-wait self-test.
#include <cstdint>

#include "ptx.cuh"
#include "registry.h"

namespace sat {

__global__ void sat_scale_kernel(float* __restrict__ C, int kind, long long rows, long long cols, long long ldc,
                                 float beta)
{
    for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
        for (long long c = threadIdx.x; c < cols; c += blockDim.x) {
            const long long i = r * ldc + c;
            c_store(C, kind, i, beta == 0.0f ? 0.0f : beta * c_load(C, kind, i));
        }
    }
}

cudaError_t launch_scale(float* C, int kind, long long rows, long long cols, long long ldc, float beta,
                         cudaStream_t stream)
{
    if (rows <= 0 || cols <= 0)
        return cudaSuccess;
    const long long blocks = rows < 8192 ? rows : 8192;
    sat_scale_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(C, kind, rows, cols, ldc, beta);
    return cudaGetLastError();
}

// Row packing for operands whose rows are not 16-byte aligned: dst row r is
// src row r (cols elements of `es` bytes, row stride ld_src), written with
// row stride ld_dst (a multiple of 16 bytes, dst 16-byte aligned) and zeros
// after the last column. Each thread writes one 16-byte piece of dst, read
// from src as aligned-down 4-byte words (elements are es-aligned, so a piece
// spans at most five words) shifted into place: copying order only, no
// arithmetic on the values. Memory-bound: one read and one write per element.
__global__ void sat_pack_rows_kernel(const uint8_t* __restrict__ src, long long ld_src_bytes, uint8_t* __restrict__ dst,
                                     long long ld_dst_bytes, long long rows, long long row_bytes)
{
    const long long pieces = ld_dst_bytes / 16;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < rows * pieces; i += stride) {
        const long long r = i / pieces, b0 = (i - r * pieces) * 16;  // byte offset of the piece within the row
        const uint8_t* row = src + r * ld_src_bytes;
        uint32_t out[4];
        if (b0 + 16 <= row_bytes) {
            // Whole piece inside the row: five aligned words cover it.
            const uintptr_t a = reinterpret_cast<uintptr_t>(row + b0);
            const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
            const uint32_t sh = static_cast<uint32_t>(a & 3u) * 8u;
            uint32_t v[5];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                v[j] = __ldg(w + j);
            v[4] = sh ? __ldg(w + 4) : 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                out[j] = sh ? __funnelshift_r(v[j], v[j + 1], sh) : v[j];
        } else {
            // The row's last piece: bytes past the row are zero.
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t word = 0;
                for (int b = 0; b < 4; ++b) {
                    const long long o = b0 + 4 * j + b;
                    if (o < row_bytes)
                        word |= static_cast<uint32_t>(__ldg(row + o)) << (8 * b);
                }
                out[j] = word;
            }
        }
        *reinterpret_cast<uint4*>(dst + r * ld_dst_bytes + b0) = make_uint4(out[0], out[1], out[2], out[3]);
    }
}

cudaError_t launch_pack_rows(const void* src, long long ld_src_bytes, void* dst, long long ld_dst_bytes,
                             long long rows, long long row_bytes, int sm_count, cudaStream_t stream)
{
    if (rows <= 0)
        return cudaSuccess;
    const long long work = rows * (ld_dst_bytes / 16);
    long long blocks = (work + 255) / 256;
    const long long cap = static_cast<long long>(sm_count) * 8;
    if (blocks > cap)
        blocks = cap;
    sat_pack_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint8_t*>(src), ld_src_bytes, static_cast<uint8_t*>(dst), ld_dst_bytes, rows, row_bytes);
    return cudaGetLastError();
}

// Split-K reduction: C[r][c] = alpha * (W_0[r][c] + W_1[r][c] + ... + W_{S-1}[r][c])
// + beta * C[r][c], summed in the fixed order s = 0, 1, ..., S-1 so that the
// result is the same on every run. W_s is slice s of the workspace (`slice`
// floats apart, rows of `cols` floats); C has row stride ldc. beta == 0 never
// reads C. Memory-bound: S + 1 (+1) floats of traffic per output element.
// Each thread takes four consecutive columns of one row, as one 16-byte
// access where the columns, the strides and C allow it.
__global__ void sat_splitk_reduce_kernel(const float* __restrict__ ws, int S, long long slice, float* C, int kind,
                                         long long rows, long long cols, long long ldc, float alpha, float beta)
{
    const long long c4 = (cols + 3) / 4;
    const bool vec = kind == 0 && cols % 4 == 0 && ldc % 4 == 0 && slice % 4 == 0 &&
                     reinterpret_cast<uintptr_t>(C) % 16 == 0;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < rows * c4; i += stride) {
        const long long r = i / c4, c = (i - r * c4) * 4;
        const float* w = ws + r * cols + c;
        if (vec) {
            float* o = C + r * ldc + c;
            float4 a = *reinterpret_cast<const float4*>(w);
            for (int s = 1; s < S; ++s) {
                const float4 b = *reinterpret_cast<const float4*>(w + s * slice);
                a.x += b.x;
                a.y += b.y;
                a.z += b.z;
                a.w += b.w;
            }
            float4 v = make_float4(alpha * a.x, alpha * a.y, alpha * a.z, alpha * a.w);
            if (beta != 0.0f) {
                const float4 x = *reinterpret_cast<const float4*>(o);
                v.x = fmaf(beta, x.x, v.x);
                v.y = fmaf(beta, x.y, v.y);
                v.z = fmaf(beta, x.z, v.z);
                v.w = fmaf(beta, x.w, v.w);
            }
            *reinterpret_cast<float4*>(o) = v;
        } else {
            for (int e = 0; e < 4 && c + e < cols; ++e) {
                float a = w[e];
                for (int s = 1; s < S; ++s)
                    a += w[s * slice + e];
                float v = alpha * a;
                const long long i = r * ldc + c + e;
                if (beta != 0.0f)
                    v = fmaf(beta, c_load(C, kind, i), v);
                c_store(C, kind, i, v);
            }
        }
    }
}

cudaError_t launch_splitk_reduce(const float* ws, int S, long long slice, float* C, int kind, long long rows,
                                 long long cols, long long ldc, float alpha, float beta, int sm_count,
                                 cudaStream_t stream)
{
    if (rows <= 0 || cols <= 0)
        return cudaSuccess;
    long long blocks = (rows * ((cols + 3) / 4) + 255) / 256;
    const long long cap = 8LL * (sm_count > 0 ? sm_count : 1);
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    sat_splitk_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(ws, S, slice, C, kind, rows, cols,
                                                                               ldc, alpha, beta);
    return cudaGetLastError();
}

// One CTA waits on a barrier that nothing arrives at, through the same
// bounded wait the GEMM kernels use; it must give up after timeout_ns and
// record the timeout bit.
__global__ void sat_wait_probe_kernel(uint32_t* err, unsigned long long timeout_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtl w{&abort_flag, err, timeout_ns};
        wait_bar<false>(smem_u32(&bar), 0, w, 1u << 4);
    }
    __syncthreads();
}

cudaError_t launch_wait_probe(uint32_t* err, unsigned long long timeout_ns, cudaStream_t stream)
{
    sat_wait_probe_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
    return cudaGetLastError();
}

const KernelEntry* find_entry(int dt, int bn, int cg, int prod, int stages)
{
    const KernelEntry* tab[3];
    int num[3];
    if (dt == kDtTF32) {
        tab[0] = kEntriesTF32, tab[1] = kEntriesTF32Alt, tab[2] = kEntriesTF32Trans;
        num[0] = kNumEntriesTF32, num[1] = kNumEntriesTF32Alt, num[2] = kNumEntriesTF32Trans;
    } else if (dt == kDtBF16) {
        tab[0] = kEntriesBF16, tab[1] = kEntriesBF16Alt, tab[2] = kEntriesBF16Trans;
        num[0] = kNumEntriesBF16, num[1] = kNumEntriesBF16Alt, num[2] = kNumEntriesBF16Trans;
    } else {
        tab[0] = kEntriesFP16, tab[1] = kEntriesFP16Alt, tab[2] = kEntriesFP16Trans;
        num[0] = kNumEntriesFP16, num[1] = kNumEntriesFP16Alt, num[2] = kNumEntriesFP16Trans;
    }
    const KernelEntry* best = nullptr;
    for (int g = 0; g < 3; ++g) {
        for (int i = 0; i < num[g]; ++i) {
            const KernelEntry& k = tab[g][i];
            if (k.bn != bn || k.cg != cg || k.prod != prod)
                continue;
            if (stages > 0 && k.stages == stages)
                return &k;
            if (stages == 0 && (!best || k.stages > best->stages))
                best = &k;
        }
    }
    return best;
}

}  // namespace sat
