"""GPU parity of transposed and strided operands (C = alpha*op(A)*op(B) +
beta*C with leading dimensions) against the FP64 oracle, through the C ABI.

The oracle takes the logical op(A) (M x K) and op(B) (K x N). The device
gets them as stored: transposed where the plan says so, with rows padded
beyond the logical width. The padding holds NaN, so a kernel that reads it
fails the comparison, and C's padding holds a sentinel that must survive.
Dyadic inputs keep every sum exact, so the comparison is bit for bit.
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

NAN_BITS = {"bf16": np.uint16(0x7FC0), "fp16": np.uint16(0x7E00)}
SENTINEL = np.float32(-12345.0)


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    sat.build()
    sat.lib()


def _stored(x, transposed, ld, dtype):
    """x (logical rows x cols) as stored: transposed or not, each stored row
    padded to ld elements with NaN."""
    s = np.ascontiguousarray(x.T if transposed else x)
    pad = np.full((s.shape[0], ld), NAN_BITS.get(dtype, np.float32(np.nan)), dtype=s.dtype)
    pad[:, :s.shape[1]] = s
    return pad


def _run(M, N, K, dtype, ta, tb, lda, ldb, ldc, config, alpha, beta, family="dyadic", seed=71):
    A, B, C0 = si.problem(M, N, K, dtype, family, seed, family)
    dA = to_dev(_stored(A, ta, lda, dtype), dtype)
    dB = to_dev(_stored(B, tb, ldb, dtype), dtype)
    Cs = np.full((M, ldc), SENTINEL, np.float32)
    Cs[:, :N] = C0
    dC = to_dev(Cs)
    with sat.Plan(M, N, K, dtype, config, trans_a=ta, trans_b=tb) as plan:
        desc = plan.describe()
        plan.run(dA, dB, dC, alpha, beta, stream(), lda=lda, ldb=ldb, ldc=ldc)
        torch.cuda.synchronize()
        sat.check(plan.status())
    out = dC.cpu().numpy()
    assert np.all(out[:, N:] == SENTINEL), f"C padding was written [{desc}]"
    return A, B, C0, out[:, :N], desc


def _ld(width, dtype, extra):
    """A row stride of at least `width` elements that is a 16-byte multiple, plus `extra` 16-byte units."""
    per16 = 4 if dtype == "tf32" else 8
    return -(-width // per16) * per16 + extra * per16


LAYOUTS = [(False, False), (True, False), (False, True), (True, True)]


@pytest.mark.parametrize("config", [None, "128,1,0,4", "256,1,1,2", "256,2,0,4", "256,2,1,2,3"])
@pytest.mark.parametrize("ta,tb", LAYOUTS, ids=lambda x: "T" if x else "N")
@pytest.mark.parametrize("dtype", ["tf32", "bf16", "fp16"])
def test_layouts_and_strides_dyadic_exact(dtype, ta, tb, config):
    M, N, K = 333, 520, 264
    lda = _ld(M if ta else K, dtype, 1)
    ldb = _ld(K if tb else N, dtype, 2)
    A, B, C0, got, desc = _run(M, N, K, dtype, ta, tb, lda, ldb, N + 12, config, 1.5, 0.5)
    assert (" ta" in desc) == ta and (" tb" in desc) == tb
    _, ref32 = oracle.gemm(A, B, C0, 1.5, 0.5, dtype)
    checks.assert_bit_exact(got, ref32, f"{dtype} ta={ta} tb={tb} [{desc}]")


@pytest.mark.parametrize("ta,tb", LAYOUTS[1:], ids=["TN", "NT", "TT"])
def test_layouts_gaussian_rel_rms(ta, tb):
    M, N, K = 700, 1000, 1100
    dtype = "bf16"
    A, B, C0, got, desc = _run(M, N, K, dtype, ta, tb, _ld(M if ta else K, dtype, 0), _ld(K if tb else N, dtype, 0),
                               N, None, 1.0, -1.0, family="normal", seed=72)
    ref64, _ = oracle.gemm(A, B, C0, 1.0, -1.0, dtype)
    checks.assert_rel_rms(got, ref64, si.REL_RMS_BOUND[dtype], desc)


@pytest.mark.parametrize("ta,tb", LAYOUTS[1:], ids=["TN", "NT", "TT"])
def test_layouts_with_stream_k(ta, tb):
    M, N, K = 1650, 3192, 632
    dtype = "bf16"
    A, B, C0, got, desc = _run(M, N, K, dtype, ta, tb, _ld(M if ta else K, dtype, 0), _ld(K if tb else N, dtype, 0),
                               N, "128,1,0,4,sk", 1.5, 0.5, seed=73)
    assert " sk" in desc
    _, ref32 = oracle.gemm(A, B, C0, 1.5, 0.5, dtype)
    checks.assert_bit_exact(got, ref32, desc)


@pytest.mark.parametrize("config", [None, "256,1,0,8,plain"])
def test_untransposed_row_strides_off_16_bytes(config):
    # Class views of A and B packed into aligned rows, or the plain loads.
    M, N, K = 150, 264, 96
    dtype = "bf16"
    A, B, C0, got, desc = _run(M, N, K, dtype, False, False, K + 1, N + 3, N + 1, config, 1.0, 1.0, seed=74)
    _, ref32 = oracle.gemm(A, B, C0, 1.0, 1.0, dtype)
    checks.assert_bit_exact(got, ref32, desc)


def test_transposed_operands_need_tma_strides():
    M, N, K = 64, 64, 64
    x = torch.zeros(64 * 80, dtype=torch.bfloat16, device="cuda")
    c = torch.zeros(64 * 64, device="cuda")
    with sat.Plan(M, N, K, "bf16", trans_a=True) as plan:
        with pytest.raises(sat.GemmError):
            plan.run(x, x, c, 1.0, 0.0, stream(), lda=65, ldb=64, ldc=64)   # 130-byte rows
        with pytest.raises(sat.GemmError):
            plan.run(x, x, c, 1.0, 0.0, stream(), lda=32, ldb=64, ldc=64)   # below M


def test_k_zero_scales_strided_c():
    M, N = 40, 50
    C0 = si.c_matrix("normal", M, N, 3)
    Cs = np.full((M, N + 6), SENTINEL, np.float32)
    Cs[:, :N] = C0
    dC = to_dev(Cs)
    with sat.Plan(M, N, 0, "tf32") as plan:
        plan.run(0, 0, dC, 1.0, 0.25, stream(), ldc=N + 6)
        torch.cuda.synchronize()
    out = dC.cpu().numpy()
    assert np.array_equal(out[:, :N], (0.25 * C0.astype(np.float64)).astype(np.float32))
    assert np.all(out[:, N:] == SENTINEL)


def _c16(x, c_type):
    """fp32 values rounded to the 16-bit C type (nearest, ties to even), as bit patterns."""
    if c_type == "bf16":
        return si.f32_to_bf16_bits(x.astype(np.float32))
    return x.astype(np.float32).astype(np.float16).view(np.uint16)


# 16-bit C: the epilogue reads C in that type (beta != 0), computes in fp32
# and rounds once. Dyadic C0 is exact in both 16-bit types; the fp32 result
# is exact, so rounding it once must give the oracle's value rounded once.
@pytest.mark.parametrize("config", [None, "256,2,0,4", "128,1,1,2,3", "64,1,0,4,swap"])
@pytest.mark.parametrize("c_type", ["bf16", "fp16"])
@pytest.mark.parametrize("dtype", ["tf32", "bf16"])
def test_16_bit_c_dyadic(dtype, c_type, config):
    M, N, K = 333, 520, 264
    if config and "swap" in config:
        M = 27
    A, B, C0 = si.problem(M, N, K, dtype, "dyadic", 81, "dyadic")
    _, ref32 = oracle.gemm(A, B, C0, 1.5, 0.5, dtype)
    ldc = N + 8
    Cs = np.full((M, ldc), 0x1234, np.uint16)
    Cs[:, :N] = _c16(C0, c_type)
    dC = torch.from_numpy(Cs).cuda()
    with sat.Plan(M, N, K, dtype, config, c_type=c_type) as plan:
        desc = plan.describe()
        assert f" c{c_type}" in desc
        plan.run(to_dev(A, dtype), to_dev(B, dtype), dC, 1.5, 0.5, stream(), ldc=ldc)
        torch.cuda.synchronize()
        sat.check(plan.status())
    out = dC.cpu().numpy()
    assert np.all(out[:, N:] == 0x1234), f"C padding was written [{desc}]"
    assert np.array_equal(out[:, :N], _c16(ref32, c_type)), f"{dtype} -> {c_type} [{desc}]"


def test_16_bit_c_with_k_zero_scales_in_place():
    M, N = 20, 30
    C0 = si.c_matrix("dyadic", M, N, 5)
    dC = torch.from_numpy(_c16(C0, "bf16")).cuda()
    with sat.Plan(M, N, 0, "bf16", c_type="bf16") as plan:
        plan.run(0, 0, dC, 1.0, 0.5, stream())
        torch.cuda.synchronize()
    assert np.array_equal(dC.cpu().numpy(), _c16(0.5 * C0, "bf16"))


# Class-view tiles write fp32 C rows in 16-byte stores when the rows P apart
# lie a whole number of 16-byte units apart: each chunk's 16-byte-aligned
# columns as whole units, and the columns at the chunk's two ends (sharing
# 16-byte units with the neighbouring chunks) element by element.
# C sits coff floats into its allocation with row stride N + dldc; every
# float around it holds a sentinel that must survive. K = 131 gives P = 4
# (tf32) or 8 (bf16), where every ldc qualifies; K = 130 (tf32) and 132
# (bf16) give P = 2, where odd ldc keeps the element-wise row stores.
@pytest.mark.parametrize("K", [131, 130, 132])
@pytest.mark.parametrize("coff", [0, 3])
@pytest.mark.parametrize("dldc", [0, 1, 3])
@pytest.mark.parametrize("config", [None, "128,1,0,4", "256,1,1,2"])
@pytest.mark.parametrize("dtype", ["tf32", "bf16"])
def test_class_view_c_boxes_and_edge_columns(dtype, config, dldc, coff, K):
    M, N = 700, 600
    A, B, C0 = si.problem(M, N, K, dtype, "dyadic", 95, "dyadic")
    _, ref32 = oracle.gemm(A, B, C0, 1.5, 0.5, dtype)
    ldc = N + dldc
    Cs = np.full(coff + M * ldc + 8, SENTINEL, np.float32)
    Cs[coff:coff + M * ldc].reshape(M, ldc)[:, :N] = C0
    dC = to_dev(Cs)
    with sat.Plan(M, N, K, dtype, config) as plan:
        desc = plan.describe()
        plan.run(to_dev(A, dtype), to_dev(B, dtype), dC.data_ptr() + 4 * coff, 1.5, 0.5, stream(), ldc=ldc)
        torch.cuda.synchronize()
        sat.check(plan.status())
    out = dC.cpu().numpy()
    view = out[coff:coff + M * ldc].reshape(M, ldc)
    assert np.all(out[:coff] == SENTINEL) and np.all(out[coff + M * ldc:] == SENTINEL), f"outside C [{desc}]"
    assert np.all(view[:, N:] == SENTINEL), f"C padding was written [{desc}]"
    checks.assert_bit_exact(view[:, :N], ref32, f"{dtype} K {K} ldc {ldc} offset {coff} [{desc}]")
