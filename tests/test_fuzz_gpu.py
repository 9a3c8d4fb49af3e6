"""Seeded random problems through the C ABI, bit-exact against the oracle.

Each case draws a dtype, a shape with ragged tails, a forced configuration
(or the dispatcher's), row strides, pointer offsets that put A, B and C off
16-byte boundaries, and alpha and beta. The inputs are the dyadic family, so
the result is exact and unique: any slip in an index, a tail, a class view,
a packing, a K split or stream-K piece, or the epilogue shows as a changed
bit. The padding after each row of A and B holds NaN (a kernel that reads it
fails), and every float around C holds a sentinel that must survive.
"""
import numpy as np
import pytest
import torch

import oracle
import shape_adaptive_tile_gb300 as sat
import synth_inputs as si
from tests import checks
from tests.gpu_util import stream

pytestmark = pytest.mark.gpu

NAN_BITS = {"bf16": np.uint16(0x7FC0), "fp16": np.uint16(0x7E00)}
SENTINEL = np.float32(-12345.0)
CONFIGS = [None, "256,2,0,4", "256,2,1,8", "128,2,0,2", "128,1,1,2", "256,1,0,8", "64,1,0,4", "128,1,0,4,st4",
           "256,2,0,4,sk", "128,1,1,2,sk", "128,1,0,4,2", "256,1,0,2,3", "128,1,0,4,plain", "256,2,0,4,fwd",
           "128,1,0,4,cload"]
SWAP_CONFIGS = ["64,1,0,2,swap", "32,1,1,2,swap", "128,1,0,8,swap"]


def _case(i):
    rng = np.random.default_rng(2026 + i)
    dtype = ("tf32", "bf16", "fp16")[i % 3]
    skinny = i % 8 == 7
    M = int(rng.integers(1, 129)) if skinny else int(rng.integers(1, 1300))
    N = int(rng.integers(1, 1300))
    K = int(rng.integers(1, 600))
    config = SWAP_CONFIGS[(i // 8) % len(SWAP_CONFIGS)] if skinny else CONFIGS[int(rng.integers(0, len(CONFIGS)))]
    pad = [int(rng.integers(0, 6)) for _ in range(3)]
    off = [int(rng.integers(0, 4)) for _ in range(3)]
    alpha = float(rng.choice([1.0, 1.5, -0.5]))
    beta = float(rng.choice([0.0, 0.5, -1.0]))
    return dtype, M, N, K, config, pad, off, alpha, beta


def _stored(x, ld, off, dtype):
    """x's rows padded to ld with NaN, after `off` NaN elements."""
    nan = NAN_BITS.get(dtype, np.float32(np.nan))
    flat = np.full(off + x.shape[0] * ld + 8, nan, dtype=x.dtype)
    flat[off:off + x.shape[0] * ld].reshape(x.shape[0], ld)[:, :x.shape[1]] = x
    return flat


@pytest.mark.parametrize("i", range(256))
def test_random_problem_bit_exact(i):
    dtype, M, N, K, config, pad, off, alpha, beta = _case(i)
    A, B, C0 = si.problem(M, N, K, dtype, "dyadic", 300 + i, "dyadic")
    _, ref32 = oracle.gemm(A, B, C0, alpha, beta, dtype)
    lda, ldb, ldc = K + pad[0], N + pad[1], N + pad[2]
    es = 4 if dtype == "tf32" else 2
    tdt = {"tf32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    fa, fb = _stored(A, lda, off[0], dtype), _stored(B, ldb, off[1], dtype)
    dA = torch.from_numpy(fa).cuda() if dtype != "bf16" else torch.from_numpy(fa).view(torch.bfloat16).cuda()
    dB = torch.from_numpy(fb).cuda() if dtype != "bf16" else torch.from_numpy(fb).view(torch.bfloat16).cuda()
    assert dA.dtype == tdt and dB.dtype == tdt
    Cs = np.full(off[2] + M * ldc + 8, SENTINEL, np.float32)
    Cs[off[2]:off[2] + M * ldc].reshape(M, ldc)[:, :N] = C0
    dC = torch.from_numpy(Cs).cuda()
    what = f"{dtype} M={M} N={N} K={K} config={config} lds={lda},{ldb},{ldc} offsets={off} alpha={alpha} beta={beta}"
    with sat.Plan(M, N, K, dtype, config) as plan:
        desc = plan.describe()
        plan.run(dA.data_ptr() + es * off[0], dB.data_ptr() + es * off[1], dC.data_ptr() + 4 * off[2], alpha, beta,
                 stream(), lda=lda, ldb=ldb, ldc=ldc)
        torch.cuda.synchronize()
        sat.check(plan.status())
    out = dC.cpu().numpy()
    view = out[off[2]:off[2] + M * ldc].reshape(M, ldc)
    assert np.all(out[:off[2]] == SENTINEL) and np.all(out[off[2] + M * ldc:] == SENTINEL), f"outside C: {what} [{desc}]"
    assert np.all(view[:, N:] == SENTINEL), f"C padding written: {what} [{desc}]"
    checks.assert_bit_exact(view[:, :N], ref32, f"{what} [{desc}]")


def _c16(x, c_type):
    """fp32 values rounded to the 16-bit C type (nearest, ties to even), as bit patterns."""
    if c_type == "bf16":
        return si.f32_to_bf16_bits(x.astype(np.float32))
    return x.astype(np.float32).astype(np.float16).view(np.uint16)


def _ld16(width, dtype, extra):
    """A row stride of at least `width` elements that is a 16-byte multiple, plus `extra` 16-byte units."""
    per16 = 4 if dtype == "tf32" else 8
    return -(-width // per16) * per16 + extra * per16


@pytest.mark.parametrize("i", range(96))
def test_random_layout_and_c_type_bit_exact(i):
    # Transposed operands (A stored K x M, B stored N x K; such plans read both
    # operands through TMA, so their strides are 16-byte multiples) and C in
    # fp32, bf16 or fp16 (rounded once, to nearest even, from the exact result).
    rng = np.random.default_rng(9000 + i)
    dtype = ("tf32", "bf16", "fp16")[i % 3]
    ta, tb = bool(rng.integers(0, 2)), bool(rng.integers(0, 2))
    c_type = ("fp32", "bf16", "fp16")[(i // 3) % 3]
    M, N, K = (int(rng.integers(1, 900)) for _ in range(3))
    config = [None, "128,1,0,4", "256,1,1,2", "256,2,0,4", "256,2,1,2,3", "256,2,0,8,sk"][int(rng.integers(0, 6))]
    alpha, beta = float(rng.choice([1.0, 1.5, -0.5])), float(rng.choice([0.0, 0.5, -1.0]))
    A, B, C0 = si.problem(M, N, K, dtype, "dyadic", 500 + i, "dyadic")
    _, ref32 = oracle.gemm(A, B, C0, alpha, beta, dtype)
    trans = ta or tb
    lda = _ld16(M if ta else K, dtype, int(rng.integers(0, 3))) if trans else (K + int(rng.integers(0, 5)))
    ldb = _ld16(K if tb else N, dtype, int(rng.integers(0, 3))) if trans else (N + int(rng.integers(0, 5)))
    ldc = N + int(rng.integers(0, 5))
    sa = np.ascontiguousarray(A.T if ta else A)
    sb = np.ascontiguousarray(B.T if tb else B)
    fa, fb = _stored(sa, lda, 0, dtype), _stored(sb, ldb, 0, dtype)
    to = (lambda f: torch.from_numpy(f).view(torch.bfloat16).cuda()) if dtype == "bf16" else \
        (lambda f: torch.from_numpy(f).cuda())
    dA, dB = to(fa), to(fb)
    if c_type == "fp32":
        Cs = np.full((M, ldc), SENTINEL, np.float32)
        Cs[:, :N] = C0
        expect, pad = ref32, SENTINEL
    else:
        Cs = np.full((M, ldc), 0x1234, np.uint16)
        Cs[:, :N] = _c16(C0, c_type)
        expect, pad = _c16(ref32, c_type), 0x1234
    dC = torch.from_numpy(Cs).cuda()
    what = f"{dtype} M={M} N={N} K={K} ta={ta} tb={tb} C={c_type} config={config} lds={lda},{ldb},{ldc} " \
           f"alpha={alpha} beta={beta}"
    with sat.Plan(M, N, K, dtype, config, trans_a=ta, trans_b=tb, c_type=c_type) as plan:
        desc = plan.describe()
        plan.run(dA, dB, dC, alpha, beta, stream(), lda=lda, ldb=ldb, ldc=ldc)
        torch.cuda.synchronize()
        sat.check(plan.status())
    out = dC.cpu().numpy()
    assert np.all(out[:, N:] == pad), f"C padding written: {what} [{desc}]"
    assert np.array_equal(out[:, :N], expect), f"{what} [{desc}]"
