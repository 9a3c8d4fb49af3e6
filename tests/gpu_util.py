"""Helpers for the GPU tests: move seeded inputs to the device, run the C
ABI, bring results back."""
import numpy as np
import torch

import shape_adaptive_tile_gb300 as sat

TORCH_DT = {"tf32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}


def to_dev(x, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t.cuda()


def stream():
    return torch.cuda.current_stream().cuda_stream


def run(plan, dA, dB, dC, alpha, beta):
    plan.run(dA, dB, dC, alpha, beta, stream())


def run_np(M, N, K, dtype, A, B, C0, alpha, beta, config=None):
    """One GEMM through the C ABI on numpy inputs; returns (C, description)."""
    dA, dB = to_dev(A, dtype), to_dev(B, dtype)
    dC = to_dev(C0) if C0 is not None else torch.full((M, N), float("nan"), device="cuda")
    with sat.Plan(M, N, K, dtype, config) as plan:
        run(plan, dA, dB, dC, alpha, beta)
        torch.cuda.synchronize()
        sat.check(plan.status())
        desc = plan.describe()
    return dC.cpu().numpy(), desc
