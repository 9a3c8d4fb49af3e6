"""Every workload of the deterministic-GEMM study at full size, through the
C ABI with the dispatcher's own choice (the launch configuration the
benchmark times), compared with the oracle on the complete output.

The gates are the study's: bit-exact where the inputs are dyadic (here every
shape is also run with the dyadic family, where exactly one result is
correct), rel_rms over all M x N outputs within the dtype bound on the
Gaussian/uniform inputs, and identical bits over 10 runs. The reference is
the oracle's full-output form (its float64 matrix product as the sum over
k), which equals the plain ascending-k loop bit for bit on dyadic inputs
and to a few double ulps otherwise.
"""
import numpy as np
import pytest
import torch

import oracle
import shape_adaptive_tile_gb300 as sat
import synth_inputs as si
from tests import checks
from tests.gpu_util import run, to_dev

pytestmark = pytest.mark.gpu

RUNS = 10


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    sat.build()
    sat.lib()


def _run_workload(dtype, M, N, K, family, alpha, beta, c_family, seed):
    A, B, C0 = si.problem(M, N, K, dtype, family, seed, c_family)
    dA, dB = to_dev(A, dtype), to_dev(B, dtype)
    dC0 = to_dev(C0) if C0 is not None else None
    out = torch.empty(M, N, device="cuda")
    first = None
    with sat.Plan(M, N, K, dtype) as plan:
        desc = plan.describe()
        for i in range(RUNS):
            if dC0 is not None:
                out.copy_(dC0)
            else:
                out.fill_(float("nan"))        # beta == 0: C must not be read
            run(plan, dA, dB, out, alpha, beta)
            bits = out.view(torch.int32)
            if first is None:
                first = bits.clone()
            else:
                assert torch.equal(bits, first), f"run {i} differs bitwise from run 0 [{desc}]"
        torch.cuda.synchronize()
        sat.check(plan.status())
    del dA, dB, dC0, out
    got = first.view(torch.float32).cpu().numpy()
    del first
    ref64, ref32 = oracle.gemm_full(A, B, C0, alpha, beta, dtype)
    return got, ref64, ref32, desc


@pytest.mark.parametrize("w", si.WORKLOADS, ids=lambda w: f"{w[1]}-{w[0]}")
def test_workload(w):
    name, dtype, (M, N, K), family, alpha, beta, c_family, seed, gate = w
    got, ref64, ref32, desc = _run_workload(dtype, M, N, K, family, alpha, beta, c_family, seed)
    assert got.shape == (M, N)
    if gate == "exact":
        checks.assert_bit_exact(got, ref32, f"{name} {dtype} [{desc}]")
    else:
        r = checks.assert_rel_rms(got, ref64, si.REL_RMS_BOUND[dtype], f"{name} {dtype} [{desc}]")
        print(f"rel_rms {name} {dtype}: {r:.3e} over {M * N} outputs [{desc}]")


SHAPES = sorted({(w[1], w[2]) for w in si.WORKLOADS})


@pytest.mark.parametrize("dtype,shape", SHAPES, ids=lambda x: str(x))
def test_workload_shape_dyadic_exact(dtype, shape):
    M, N, K = shape
    got, _, ref32, desc = _run_workload(dtype, M, N, K, "dyadic", 1.5, 0.5, "dyadic", 100 + M % 97)
    checks.assert_bit_exact(got, ref32, f"dyadic {dtype} {shape} [{desc}]")
