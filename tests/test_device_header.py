"""The device routine's header (include/gemm_device.cuh) used the way its
comment describes, from a caller's own translation unit outside the
library: a persistent kernel of the caller's that does other work, then the
GEMM phase, then more work in the same launch. On CPU it is compiled only;
on a GPU (-m gpu) it is built into a shared library of its own, launched
with the parameters gemm_device_prepare() fills in, and its C compared with
the oracle."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

USER_SOURCE = r'''
#include <cuda_runtime.h>
#include "gemm_device.cuh"

template <int DT, int BN, int CG>
__global__ void __launch_bounds__(GemmDeviceTile<DT, BN, CG>::THREADS, 1)
    user_megakernel(const __grid_constant__ gemm_device_params p, float* flag)
{
    extern __shared__ uint8_t smem[];
    if (blockIdx.x == 0 && threadIdx.x == 0)
        flag[0] = 1.0f;                       // work before the GEMM phase
    gemm_device_run<DT, BN, CG>(p, smem);    // every thread of every block
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0)
        flag[1] = p.args.C[0];                // work after it, on this block's first tile
}

template <int DT, int BN, int CG>
static int launch(const gemm_device_params& p, float* flag, cudaStream_t s)
{
    if (cudaFuncSetAttribute(user_megakernel<DT, BN, CG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             p.smem_bytes) != cudaSuccess)
        return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(p.threads);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = p.cluster_size;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, user_megakernel<DT, BN, CG>, p, flag) == cudaSuccess ? 0 : -2;
}

extern "C" int user_params_bytes() { return static_cast<int>(sizeof(gemm_device_params)); }

// The bf16 instance gemm_device_prepare() named in the params (128 x 128 or CTA pairs of 256 x 256).
extern "C" int user_launch_bf16(const void* params, float* flag, void* stream)
{
    const gemm_device_params& p = *static_cast<const gemm_device_params*>(params);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.bn == 128 && p.cta_group == 1)
        return launch<sat::kDtBF16, 128, 1>(p, flag, s);
    if (p.bn == 256 && p.cta_group == 2)
        return launch<sat::kDtBF16, 256, 2>(p, flag, s);
    return -3;
}
'''


def _nvcc():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    return nvcc


def _build(tmp_path, shared):
    src = tmp_path / "user.cu"
    src.write_text(USER_SOURCE)
    out = tmp_path / ("libuser.so" if shared else "user.o")
    cmd = [_nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-maxrregcount=200",
           "-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(ROOT, "shape_adaptive_tile_gb300", "csrc"),
           "-Xcompiler", "-fPIC"] + (["-shared"] if shared else ["-c"]) + [str(src), "-o", str(out)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    return out


def test_device_header_compiles_in_a_user_kernel(tmp_path):
    out = _build(tmp_path, shared=False)
    assert out.stat().st_size > 0


@pytest.mark.gpu
@pytest.mark.parametrize("cta_group", [1, 2])
def test_user_kernel_runs_the_gemm_phase(tmp_path, cta_group):
    import torch
    import oracle
    import shape_adaptive_tile_gb300 as sat
    import synth_inputs as si
    from tests import checks
    from tests.gpu_util import stream, to_dev

    sat.build()
    user = ctypes.CDLL(str(_build(tmp_path, shared=True)))
    user.user_launch_bf16.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    # Ragged in M, N and K (rows of 16-byte multiples, as the routine's tensor
    # maps need); several tiles per block at 128 x 128.
    M, N, K = 1000, 712, 328
    A, B, C0 = si.problem(M, N, K, "bf16", "dyadic", 63, "dyadic")
    _, ref32 = oracle.gemm(A, B, C0, 1.5, -0.5, "bf16")
    dA, dB, dC = to_dev(A, "bf16"), to_dev(B, "bf16"), to_dev(C0)
    flag = torch.zeros(2, device="cuda")
    size = user.user_params_bytes()
    buf = (ctypes.c_uint8 * (size + 64))()
    ptr = (ctypes.addressof(buf) + 63) // 64 * 64   # the tensor maps want 64-byte alignment
    assert sat.gemm_device_prepare(M, N, K, "bf16", dA, dB, dC, 1.5, -0.5, cta_group, ptr, size) == 0, \
        sat.gemm_last_error()
    assert user.user_launch_bf16(ptr, flag.data_ptr(), stream()) == 0
    torch.cuda.synchronize()
    got = dC.cpu().numpy()
    checks.assert_bit_exact(got, ref32, f"user kernel, cta_group {cta_group}")
    f = flag.cpu().numpy()
    assert f[0] == 1.0 and f[1] == np.float32(ref32[0, 0])
