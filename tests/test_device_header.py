"""The device routine's header (include/gemm_device.cuh) compiles in a
caller's own translation unit, outside the library, with the include paths
and flags its comment gives: a persistent kernel of the caller's that runs
other work, then the GEMM phase, then more work. Compiled only (no GPU
needed); the GPU suite runs the library's own kernel built the same way."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

USER_KERNEL = r'''
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
        flag[1] = p.args.C[0];                // work after it, on this block's tiles
}

template __global__ void user_megakernel<sat::kDtBF16, 128, 1>(const __grid_constant__ gemm_device_params, float*);
template __global__ void user_megakernel<sat::kDtTF32, 256, 2>(const __grid_constant__ gemm_device_params, float*);
'''


def test_device_header_compiles_in_a_user_kernel(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = tmp_path / "user.cu"
    src.write_text(USER_KERNEL)
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-maxrregcount=200",
           "-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(ROOT, "shape_adaptive_tile_gb300", "csrc"),
           "-c", str(src), "-o", str(tmp_path / "user.o")]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    assert (tmp_path / "user.o").stat().st_size > 0
