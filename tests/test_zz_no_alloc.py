"""gemm_run_noalloc, the allocation-free entry point, through the C ABI.

It serves callers that must not allocate device memory while they run (a
framework that owns the device memory, a latency-bound loop that cannot
afford cudaFree's synchronisation, a host that forbids allocation after
start-up). It must give exactly what a plan and gemm_run give for the same
problem, and it must do so on two calls in a row: every call shares the
library's fixed scratch array, so the second call must not be disturbed by
what the first left there (its status word, its split-K partial tiles).

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes when run alone.
"""
import numpy as np
import pytest
import torch

import oracle
import shape_adaptive_tile_gb300 as sat
import synth_inputs as si
from tests import checks
from tests.gpu_util import stream, to_dev

pytestmark = pytest.mark.gpu

# dtype, M, N, K, family, alpha, beta
CASES = [
    ("bf16", 256, 4096, 8192, "dyadic", 1.5, 0.5),   # CTA pairs, K split 2 ways: partial tiles in the scratch
    ("tf32", 128, 2048, 16384, "normal", 1.0, 0.0),  # K split 4 ways, beta 0 (C starts as NaN, never read)
    ("tf32", 300, 260, 200, "normal", 1.0, 0.0),     # no split: only the status word is scratch
    ("fp16", 513, 264, 130, "dyadic", 1.0, 1.0),
    ("bf16", 333, 517, 389, "uniform", 1.5, 0.5),    # misaligned row strides: plain-load producer
    ("bf16", 6144, 6144, 4096, "normal", 1.0, 0.0),  # stream-K: partial tiles and counters in the scratch
    ("bf16", 16, 8192, 8192, "dyadic", 1.5, 0.5),    # skinny M: operands swapped, K split in the scratch
]


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    sat.build()
    sat.lib()


def _fresh_c(C0, M, N):
    if C0 is None:
        return torch.full((M, N), float("nan"), device="cuda")
    return to_dev(C0)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}")
def test_noalloc_matches_gemm_run_on_two_calls(case):
    dtype, M, N, K, family, alpha, beta = case
    A, B, C0 = si.problem(M, N, K, dtype, family, 21, "normal" if beta != 0 else None)
    dA, dB = to_dev(A, dtype), to_dev(B, dtype)
    ref = _fresh_c(C0, M, N)
    with sat.Plan(M, N, K, dtype) as plan:
        desc = plan.describe()
        plan.run(dA, dB, ref, alpha, beta, stream())
        torch.cuda.synchronize()
        sat.check(plan.status())
    ref_np = ref.cpu().numpy()
    ref64, ref32 = oracle.gemm(A, B, C0, alpha, beta, dtype)
    for call in range(2):
        out = _fresh_c(C0, M, N)
        rc = sat.gemm_run_noalloc(M, N, K, dtype, dA, dB, out, alpha, beta, stream())
        assert rc == 0, sat.gemm_last_error()
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        # TMA-readable rows: the same kernel, choice and K order as gemm_run,
        # so the same bits. Rows that TMA cannot address: a plan reads them
        # through class views (B packed into a copy it allocates), this entry
        # point through plain loads; the K order then differs, and the two
        # agree within the dtype's tolerance (bit for bit on dyadic inputs).
        es = 4 if dtype == "tf32" else 2
        if (K * es) % 16 == 0 and (N * es) % 16 == 0 or family == "dyadic":
            checks.assert_bit_exact(got, ref_np, f"gemm_run_noalloc call {call + 1} vs gemm_run [{desc}]")
        else:
            checks.assert_rel_rms(got, ref_np.astype(np.float64), si.REL_RMS_BOUND[dtype],
                                  f"gemm_run_noalloc call {call + 1} vs gemm_run [{desc}]")
        # And the oracle's result: exactly where the inputs are dyadic (one
        # correct answer), within the dtype's rel_rms bound otherwise.
        if family == "dyadic":
            checks.assert_bit_exact(got, ref32, f"gemm_run_noalloc call {call + 1} vs oracle [{desc}]")
        else:
            checks.assert_rel_rms(got, ref64, si.REL_RMS_BOUND[dtype],
                                  f"gemm_run_noalloc call {call + 1} vs oracle [{desc}]")


def _split_workspace_bytes(M, N, K, dtype):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    bn, cg, _, _, splits, _, _, swap, _, _ = sat.gemm_select_config(M, N, K, dtype, sms, True).split(",")
    rows = 128 * int(cg)
    return int(splits), int(splits) * (-(-M // rows) * rows) * N * 4


@pytest.mark.parametrize("dtype,M,N,K", [("bf16", 256, 4096, 8192), ("tf32", 128, 2048, 16384)])
def test_noalloc_cases_really_split_k_within_the_scratch(dtype, M, N, K):
    splits, ws = _split_workspace_bytes(M, N, K, dtype)
    assert splits > 1 and ws <= (32 << 20) - 4096


def test_noalloc_case_really_uses_stream_k():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert sat.gemm_select_config(6144, 6144, 4096, "bf16", sms, True).split(",")[6] == "1"


def test_noalloc_works_after_a_rejected_call():
    # A bad call (here a NULL operand) is rejected before any launch, and
    # the entry point still works afterwards.
    c = torch.zeros(64 * 64, device="cuda")
    assert sat.gemm_run_noalloc(64, 64, 64, "bf16", None, None, c, 1.0, 0.0, stream()) == -1
    A, B, _ = si.problem(64, 64, 64, "bf16", "dyadic", 3)
    out = torch.empty(64, 64, device="cuda")
    assert sat.gemm_run_noalloc(64, 64, 64, "bf16", to_dev(A, "bf16"), to_dev(B, "bf16"), out, 1.0, 0.0,
                                stream()) == 0
    torch.cuda.synchronize()
    _, ref32 = oracle.gemm(A, B, None, 1.0, 0.0, "bf16")
    checks.assert_bit_exact(out.cpu().numpy(), ref32, "after a rejected call")


def test_noalloc_argument_errors():
    x = torch.zeros(16, device="cuda")
    assert sat.gemm_run_noalloc(-1, 4, 4, "tf32", x, x, x, 1.0, 0.0, stream()) == -1
    assert sat.gemm_run_noalloc(4, 4, 4, "tf32", x, x, None, 1.0, 0.0, stream()) == -1
    assert sat.gemm_run_noalloc(4, 4, 4, "tf32", x, x, x.data_ptr() + 2, 1.0, 0.0, stream()) == -3
    assert sat.gemm_run_noalloc(0, 4, 4, "tf32", None, None, None, 1.0, 0.0, stream()) == 0


@pytest.mark.parametrize("i", range(32))
def test_noalloc_random_problems_bit_exact(i):
    # Seeded random shapes and operand offsets (dense strides), dyadic inputs:
    # the oracle's bits, twice in a row from the same fixed scratch.
    rng = np.random.default_rng(4000 + i)
    dtype = ("tf32", "bf16", "fp16")[i % 3]
    M = int(rng.integers(1, 128)) if i % 5 == 4 else int(rng.integers(1, 2500))
    N, K = int(rng.integers(1, 2500)), int(rng.integers(1, 3000))
    alpha, beta = float(rng.choice([1.0, 1.5])), float(rng.choice([0.0, 0.5]))
    off = int(rng.integers(0, 2))
    A, B, C0 = si.problem(M, N, K, dtype, "dyadic", 600 + i, "dyadic")
    _, ref32 = oracle.gemm(A, B, C0, alpha, beta, dtype)
    es = 4 if dtype == "tf32" else 2
    fa = np.concatenate([np.zeros(off, A.dtype), A.ravel()])
    fb = np.concatenate([np.zeros(off, B.dtype), B.ravel()])
    dA, dB = to_dev(fa, dtype), to_dev(fb, dtype)
    for call in range(2):
        out = to_dev(C0)
        rc = sat.gemm_run_noalloc(M, N, K, dtype, dA.data_ptr() + es * off, dB.data_ptr() + es * off, out, alpha,
                                  beta, stream())
        assert rc == 0, sat.gemm_last_error()
        torch.cuda.synchronize()
        checks.assert_bit_exact(out.cpu().numpy(), ref32,
                                f"noalloc call {call + 1}: {dtype} {M}x{N}x{K} offset {off} alpha {alpha} beta {beta}")
