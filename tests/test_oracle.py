"""Pins for the FP64 CPU oracle, against facts other than the oracle itself.

Each pin is chosen so that a plausible slip in the oracle fails at least one
of them: a dropped or extra k term (all-ones = K, sum of squares), a wrong
index or a transposed operand (non-square brute force, permutations, the
1x2x3 worked example), a wrong sign or a lost alpha/beta term (alpha/beta
closed forms), a wrong type decode (every fp16/bf16 bit pattern against
numpy), and a wrong final rounding (ties-to-even cases).
"""
import itertools
import os

import numpy as np
import pytest

import oracle
import synth_inputs as si
from tests import checks

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.txt")


def _exact(dtype, v):
    """Store float values exactly in the operand type of ``dtype``."""
    v = np.asarray(v, dtype=np.float64)
    s = si.store(v, dtype)
    back = {"tf32": lambda x: x.astype(np.float64),
            "fp16": lambda x: x.astype(np.float64),
            "bf16": lambda x: si.bf16_bits_to_f32(x).astype(np.float64)}[dtype](s)
    assert np.array_equal(back, v), "test value not exact in the storage type"
    return s


# --- element decoding --------------------------------------------------------

def test_decode_fp16_every_pattern_matches_numpy():
    bits = np.arange(1 << 16, dtype=np.uint32)
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle.decode("fp16", int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_decode_bf16_every_pattern_matches_fp32_widening():
    bits = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (bits << np.uint32(16)).view(np.float32).astype(np.float64)
    got = np.array([oracle.decode("bf16", int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("dtype,bits,value", [
    ("fp16", 0x3C00, 1.0), ("fp16", 0x7BFF, 65504.0), ("fp16", 0x0001, 2.0 ** -24),
    ("fp16", 0x0400, 2.0 ** -14), ("fp16", 0xC000, -2.0), ("fp16", 0x3555, 0.333251953125),
    ("bf16", 0x3F80, 1.0), ("bf16", 0x4049, 3.140625), ("bf16", 0x0001, 2.0 ** -133),
    ("bf16", 0x7F7F, (2 - 2.0 ** -7) * 2.0 ** 127), ("bf16", 0xBF00, -0.5),
    ("tf32", 0x3F800000, 1.0), ("tf32", 0x00000001, 2.0 ** -149),
])
def test_decode_known_patterns(dtype, bits, value):
    assert oracle.decode(dtype, bits) == value


# --- worked examples (tests/golden) -------------------------------------------

def _golden_cases():
    cases, cur = [], None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
            elif key == "end":
                cases.append(cur)
                cur = None
            else:
                cur[key] = vals
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_worked_example(case):
    dtype = case["dtype"][0]
    M, N, K = (int(x) for x in case["shape"])
    alpha, beta = float(case["alpha"][0]), float(case["beta"][0])
    if "Abits" in case:
        A = np.array([int(x, 16) for x in case["Abits"]], dtype=np.uint16).reshape(M, K)
        B = np.array([int(x, 16) for x in case["Bbits"]], dtype=np.uint16).reshape(K, N)
        if dtype == "fp16":
            A, B = A.view(np.float16), B.view(np.float16)
    else:
        A = _exact(dtype, [float(x) for x in case["A"]]).reshape(M, K)
        B = _exact(dtype, [float(x) for x in case["B"]]).reshape(K, N)
    C0 = np.array([float(x) for x in case["C0"]], dtype=np.float32).reshape(M, N) if "C0" in case else None
    c64, c32 = oracle.gemm(A, B, C0, alpha, beta, dtype)
    want64 = np.array([float(x) for x in case["C64"]]).reshape(M, N)
    assert np.array_equal(c64, want64)
    if "C32" in case:
        want32 = np.array([int(x, 16) for x in case["C32"]], dtype=np.uint32)
        assert np.array_equal(c32.ravel().view(np.uint32), want32)
    else:
        assert np.array_equal(c32, want64.astype(np.float32))


# --- closed forms -------------------------------------------------------------

DTYPES = ["tf32", "bf16", "fp16"]


@pytest.mark.parametrize("dtype", DTYPES)
def test_identity_both_sides(dtype):
    A = si.matrix("dyadic", dtype, 13, 9, 11, 0)
    B = si.matrix("dyadic", dtype, 9, 7, 11, 1)
    I9 = _exact(dtype, np.eye(9)).reshape(9, 9)
    I13 = _exact(dtype, np.eye(13)).reshape(13, 13)
    dec = (lambda x: si.bf16_bits_to_f32(x)) if dtype == "bf16" else (lambda x: x)
    c64, _ = oracle.gemm(A, I9, dtype=dtype)
    assert np.array_equal(c64, dec(A).astype(np.float64))
    c64, _ = oracle.gemm(I13, A, dtype=dtype)
    assert np.array_equal(c64, dec(A).astype(np.float64))
    c64, _ = oracle.gemm(I9, B, dtype=dtype)
    assert np.array_equal(c64, dec(B).astype(np.float64))


def test_permutation_rows():
    rng = np.random.default_rng(5)
    sigma = rng.permutation(17)
    P = np.zeros((17, 17))
    P[np.arange(17), sigma] = 1.0
    B = si.matrix("normal", "tf32", 17, 6, 5, 1)
    c64, _ = oracle.gemm(P.astype(np.float32), B)
    assert np.array_equal(c64, B[sigma].astype(np.float64))


@pytest.mark.parametrize("dtype", DTYPES)
def test_rank1_outer_product(dtype):
    u = si.matrix("dyadic", dtype, 23, 1, 2, 0)
    v = si.matrix("dyadic", dtype, 1, 19, 2, 1)
    dec = (lambda x: si.bf16_bits_to_f32(x)) if dtype == "bf16" else (lambda x: x)
    c64, c32 = oracle.gemm(u, v, dtype=dtype)
    want = np.outer(dec(u).astype(np.float64), dec(v).astype(np.float64))
    assert np.array_equal(c64, want)
    assert np.array_equal(c32, want.astype(np.float32))


@pytest.mark.parametrize("dtype,K", [("tf32", 1), ("tf32", 777), ("bf16", 4096), ("fp16", 2048)])
def test_all_ones_sum_equals_K(dtype, K):
    A = _exact(dtype, np.ones(3 * K)).reshape(3, K)
    B = _exact(dtype, np.ones(K * 5)).reshape(K, 5)
    c64, c32 = oracle.gemm(A, B, dtype=dtype)
    assert np.all(c64 == K) and np.all(c32 == K)


def test_sum_of_squares_closed_form():
    K = 1000
    a = np.arange(1, K + 1, dtype=np.float32)
    c64, c32 = oracle.gemm(a.reshape(1, K), a.reshape(K, 1))
    assert c64[0, 0] == K * (K + 1) * (2 * K + 1) // 6
    assert c32[0, 0] == np.float32(K * (K + 1) * (2 * K + 1) // 6)


def test_alpha_zero_gives_beta_c0():
    A, B, C0 = si.problem(9, 11, 5, "tf32", "normal", 8, "normal")
    c64, _ = oracle.gemm(A, B, C0, 0.0, 0.75)
    assert np.array_equal(c64, 0.75 * C0.astype(np.float64))


def test_alpha_scales_and_beta_zero_ignores_nan_c0():
    A, B, _ = si.problem(12, 10, 33, "tf32", "dyadic", 9)
    one, _ = oracle.gemm(A, B, None, 1.0, 0.0)
    nanC = np.full((12, 10), np.nan, dtype=np.float32)
    two, two32 = oracle.gemm(A, B, nanC, 2.0, 0.0)
    assert np.array_equal(two, 2.0 * one)
    assert np.all(np.isfinite(two32))


def test_beta_term_sign_and_scale():
    A, B, C0 = si.problem(4, 6, 3, "tf32", "dyadic", 10, "dyadic")
    ab, _ = oracle.gemm(A, B)
    c64, _ = oracle.gemm(A, B, C0, 1.5, -0.5)
    assert np.array_equal(c64, 1.5 * ab - 0.5 * C0.astype(np.float64))


def test_block_diagonal_blocks_are_independent():
    A1 = si.matrix("dyadic", "tf32", 5, 4, 12, 0)
    A2 = si.matrix("dyadic", "tf32", 3, 6, 12, 1)
    B1 = si.matrix("dyadic", "tf32", 4, 7, 12, 2)
    B2 = si.matrix("dyadic", "tf32", 6, 2, 12, 3)
    A = np.zeros((8, 10), np.float32)
    A[:5, :4], A[5:, 4:] = A1, A2
    B = np.zeros((10, 9), np.float32)
    B[:4, :7], B[4:, 7:] = B1, B2
    c, _ = oracle.gemm(A, B)
    c1, _ = oracle.gemm(A1, B1)
    c2, _ = oracle.gemm(A2, B2)
    assert np.array_equal(c[:5, :7], c1) and np.array_equal(c[5:, 7:], c2)
    assert not c[:5, 7:].any() and not c[5:, :7].any()


# --- brute force on tiny shapes ----------------------------------------------

def _naive(A, B, C0, alpha, beta):
    M, K = A.shape
    N = B.shape[1]
    out = np.empty((M, N))
    for i in range(M):
        for j in range(N):
            acc = 0.0
            for k in range(K):
                acc = acc + float(A[i, k]) * float(B[k, j])
            v = alpha * acc
            if beta != 0.0:
                v = v + beta * float(C0[i, j])
            out[i, j] = v
    return out


def test_bruteforce_all_tiny_shapes():
    seed = 0
    for M, N, K in itertools.product(range(1, 8), repeat=3):
        seed += 1
        A, B, C0 = si.problem(M, N, K, "tf32", "normal", 1000 + seed, "normal")
        c64, c32 = oracle.gemm(A, B, C0, 1.25, -0.5)
        want = _naive(A, B, C0, 1.25, -0.5)
        assert np.array_equal(c64, want), (M, N, K)
        assert np.array_equal(c32, want.astype(np.float32)), (M, N, K)
        lib = 1.25 * (A.astype(np.float64) @ B.astype(np.float64)) - 0.5 * C0.astype(np.float64)
        scale = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64)) * 1.25 + 0.5 * np.abs(C0)
        assert np.all(np.abs(c64 - lib) <= 1e-14 * scale + 1e-300), (M, N, K)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_bruteforce_16bit(dtype):
    A, B, C0 = si.problem(6, 5, 9, dtype, "normal", 77, "normal")
    dec = (lambda x: si.bf16_bits_to_f32(x)) if dtype == "bf16" else (lambda x: x)
    c64, _ = oracle.gemm(A, B, C0, 0.5, 2.0, dtype)
    assert np.array_equal(c64, _naive(dec(A), dec(B), C0, 0.5, 2.0))


# --- invariants ---------------------------------------------------------------

def test_linearity_in_B_is_exact_on_dyadic():
    A = si.matrix("dyadic", "tf32", 31, 64, 20, 0)
    B1 = si.matrix("dyadic", "tf32", 64, 29, 20, 1)
    B2 = si.matrix("dyadic", "tf32", 64, 29, 20, 2)
    c, _ = oracle.gemm(A, B1 + B2)
    c1, _ = oracle.gemm(A, B1)
    c2, _ = oracle.gemm(A, B2)
    assert np.array_equal(c, c1 + c2)


def test_dyadic_exact_in_fp32_at_largest_K():
    K = 8192
    A = _exact("tf32", np.full(2 * K, 4.0)).reshape(2, K)
    A[1, ::2] = -4.0
    B = _exact("tf32", np.full(K * 3, -4.0)).reshape(K, 3)
    c64, c32 = oracle.gemm(A, B, None, 1.5, 0.0)
    assert c64[0, 0] == -16 * K * 1.5 and c64[1, 0] == 0.0
    Ad, Bd, C0 = si.problem(3, 4, K, "tf32", "dyadic", 21, "dyadic")
    c64, c32 = oracle.gemm(Ad, Bd, C0, 1.5, 0.5)
    assert np.array_equal(c32.astype(np.float64), c64)


def test_entries_and_row_ranges_match_full():
    A, B, C0 = si.problem(37, 53, 41, "bf16", "uniform", 4, "normal")
    full64, full32 = oracle.gemm(A, B, C0, 1.5, 0.5, "bf16")
    rng = np.random.default_rng(0)
    r = rng.integers(0, 37, 200)
    c = rng.integers(0, 53, 200)
    e64, e32 = oracle.gemm_entries(A, B, r, c, C0, 1.5, 0.5, "bf16")
    assert np.array_equal(e64, full64[r, c]) and np.array_equal(e32, full32[r, c])
    p64, _ = oracle.gemm(A, B, C0, 1.5, 0.5, "bf16", row_begin=10, row_end=25)
    assert np.array_equal(p64, full64[10:25])


def test_k_zero_gives_beta_c0_and_empty_shapes():
    C0 = si.c_matrix("normal", 3, 4, 1)
    c64, _ = oracle.gemm(np.zeros((3, 0), np.float32), np.zeros((0, 4), np.float32), C0, 2.0, 0.5)
    assert np.array_equal(c64, 0.5 * C0.astype(np.float64))
    c64, _ = oracle.gemm(np.zeros((0, 5), np.float32), np.zeros((5, 4), np.float32))
    assert c64.shape == (0, 4)


def test_rejects_bad_operand_types():
    with pytest.raises(TypeError):
        oracle.gemm(np.zeros((2, 2), np.float64), np.zeros((2, 2), np.float64))
    with pytest.raises(ValueError):
        oracle.gemm(np.zeros((2, 3), np.float32), np.zeros((2, 3), np.float32))


# --- the acceptance checks reject planted mistakes ----------------------------

def test_checks_reject_one_flipped_mantissa_bit():
    A, B, _ = si.problem(16, 16, 64, "tf32", "dyadic", 0)
    _, c32 = oracle.gemm(A, B)
    bad = c32.copy()
    bad.view(np.uint32)[3, 5] ^= np.uint32(1)
    assert checks.bit_exact_mismatches(c32, c32) == 0
    assert checks.bit_exact_mismatches(bad, c32) == 1


def test_checks_reject_wrong_seed_and_nan():
    A, B, _ = si.problem(32, 32, 256, "tf32", "normal", 1)
    ref64, ref32 = oracle.gemm(A, B)
    A2, B2, _ = si.problem(32, 32, 256, "tf32", "normal", 2)
    _, other = oracle.gemm(A2, B2)
    assert oracle.rel_rms(other, ref64) > 0.5
    with pytest.raises(AssertionError):
        checks.assert_rel_rms(other, ref64, 1e-3)
    nan = ref32.copy()
    nan[0, 0] = np.nan
    with pytest.raises(AssertionError):
        checks.assert_rel_rms(nan, ref64, 1e-3)
    assert checks.bit_exact_mismatches(nan, ref32) == 1


def test_rel_rms_definition_on_a_known_case():
    ref = np.array([3.0, 4.0])
    assert oracle.rel_rms(np.array([3.0, 4.0]), ref) == 0.0
    assert oracle.rel_rms(np.array([3.0, 4.5]), ref) == pytest.approx(0.5 / 5.0, rel=1e-15)


def test_oracle_uses_unrounded_fp32_not_tf32():
    # 1 + 2^-20 carries bits below tf32's 10-bit mantissa; the oracle keeps them.
    a = np.array([[1.0 + 2.0 ** -20]], dtype=np.float32)
    c64, _ = oracle.gemm(a, np.array([[1.0]], np.float32))
    assert c64[0, 0] == 1.0 + 2.0 ** -20


# --- the full-output form (numpy's float64 product as the sum over k) ---------

def test_full_form_decodes_every_bf16_and_fp16_pattern():
    # A column of every finite pattern times [[1]] returns each value exactly.
    for dtype in ("bf16", "fp16"):
        bits = np.arange(1 << 16, dtype=np.uint32)
        want = np.array([oracle.decode(dtype, int(b)) for b in bits])
        keep = np.isfinite(want)
        col = bits[keep].astype(np.uint16).reshape(-1, 1)
        if dtype == "fp16":
            col = col.view(np.float16)
        one = _exact(dtype, [1.0]).reshape(1, 1)
        c64, _ = oracle.gemm_full(col, one, dtype=dtype)
        assert np.array_equal(c64[:, 0], want[keep])


@pytest.mark.parametrize("dtype", DTYPES)
def test_full_form_closed_forms(dtype):
    A = si.matrix("dyadic", dtype, 13, 9, 11, 0)
    I9 = _exact(dtype, np.eye(9)).reshape(9, 9)
    dec = (lambda x: si.bf16_bits_to_f32(x)) if dtype == "bf16" else (lambda x: x)
    c64, _ = oracle.gemm_full(A, I9, dtype=dtype)
    assert np.array_equal(c64, dec(A).astype(np.float64))
    K = 777
    ones_a = _exact(dtype, np.ones(3 * K)).reshape(3, K)
    ones_b = _exact(dtype, np.ones(K * 5)).reshape(K, 5)
    c64, c32 = oracle.gemm_full(ones_a, ones_b, dtype=dtype)
    assert np.all(c64 == K) and np.all(c32 == K)
    u = si.matrix("dyadic", dtype, 23, 1, 2, 0)
    v = si.matrix("dyadic", dtype, 1, 19, 2, 1)
    c64, _ = oracle.gemm_full(u, v, dtype=dtype)
    assert np.array_equal(c64, np.outer(dec(u).astype(np.float64), dec(v).astype(np.float64)))


def test_full_form_alpha_beta_terms():
    A, B, C0 = si.problem(9, 11, 5, "tf32", "dyadic", 8, "dyadic")
    ab, _ = oracle.gemm_full(A, B)
    c64, _ = oracle.gemm_full(A, B, C0, 1.5, -0.5)
    assert np.array_equal(c64, 1.5 * ab - 0.5 * C0.astype(np.float64))
    c64, _ = oracle.gemm_full(A, B, C0, 0.0, 0.75)
    assert np.array_equal(c64, 0.75 * C0.astype(np.float64))
    nan = np.full((9, 11), np.nan, np.float32)
    c64, c32 = oracle.gemm_full(A, B, nan, 2.0, 0.0)
    assert np.array_equal(c64, 2.0 * ab) and np.all(np.isfinite(c32))
    c64, _ = oracle.gemm_full(np.zeros((3, 0), np.float32), np.zeros((0, 4), np.float32), C0[:3, :4], 2.0, 0.5)
    assert np.array_equal(c64, 0.5 * C0[:3, :4].astype(np.float64))


@pytest.mark.parametrize("dtype", DTYPES)
def test_full_form_equals_plain_loop_bit_for_bit_on_dyadic(dtype):
    # Every partial sum is exact in double, so any summation order gives the
    # same bits; non-square ragged shapes catch a transposed operand.
    for M, N, K in ((1, 1, 1), (37, 53, 41), (130, 7, 300), (5, 260, 1031)):
        A, B, C0 = si.problem(M, N, K, dtype, "dyadic", 30 + M, "dyadic")
        f64, f32 = oracle.gemm_full(A, B, C0, 1.5, 0.5, dtype)
        g64, g32 = oracle.gemm(A, B, C0, 1.5, 0.5, dtype)
        assert np.array_equal(f64, g64) and np.array_equal(f32.view(np.uint32), g32.view(np.uint32))


@pytest.mark.parametrize("dtype", DTYPES)
def test_full_form_close_to_plain_loop_on_gaussian(dtype):
    M, N, K = 67, 45, 2050
    A, B, C0 = si.problem(M, N, K, dtype, "normal", 40, "normal")
    f64, f32 = oracle.gemm_full(A, B, C0, 1.25, -0.5, dtype)
    g64, g32 = oracle.gemm(A, B, C0, 1.25, -0.5, dtype)
    dec = (lambda x: si.bf16_bits_to_f32(x)) if dtype == "bf16" else (lambda x: x)
    scale = 1.25 * (np.abs(dec(A).astype(np.float64)) @ np.abs(dec(B).astype(np.float64))) + 0.5 * np.abs(C0)
    assert np.all(np.abs(f64 - g64) <= 1e-13 * scale)
    assert oracle.rel_rms(f64, g64) < 1e-14
    # A few double ulps apart, the two round to the same floats (a tie within
    # that distance has probability of order 1e-9 per element).
    assert np.array_equal(f32.view(np.uint32), g32.view(np.uint32))
