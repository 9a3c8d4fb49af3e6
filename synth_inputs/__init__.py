"""Seeded synthetic GEMM inputs, shared by the oracle side and the CUDA side.

This module draws random numbers and rounds them to the storage types the
GEMM consumes. It holds none of the GEMM's arithmetic: no products, no sums
over K, no epilogue. Both the FP64 oracle (``oracle/``) and the CUDA path
(``shape_adaptive_tile_gb300``) are fed from here, so that each side sees
exactly the same bytes.

Generator
---------
A counter-based SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; the finaliser constants are the
published ones). Draw ``i`` of stream ``(seed, stream)`` is
``mix(seed_key + (offset + i + 1) * GOLDEN)`` with
``seed_key = mix(seed * GOLDEN + stream)``. A uniform double in [0, 1) is the
top 53 bits times 2**-53, which is exact.

Families (the workloads of the deterministic-GEMM configurations)
-----------------------------------------------------------------
``dyadic``  integers uniform on {-4, ..., 4}: ``floor(9 u) - 4``. Exact in
            fp32, tf32, bf16 and fp16, so every product and partial sum of a
            GEMM with K <= 8192 is exact in fp32.
``normal``  N(0, 1) by the Box-Muller transform (Box and Muller, 1958) in
            double, rounded to fp32 (round to nearest even) and then, for the
            16-bit types, rounded again to bf16/fp16 (round to nearest even).
``uniform`` U(-1, 1) = 2u - 1 in double, rounded the same way.

Matrices of one problem use separate streams: A = stream 0, B = stream 1,
C0 = stream 2. Values are laid out row-major.

Storage: fp32 -> ``numpy.float32``; fp16 -> ``numpy.float16``; bf16 ->
``numpy.uint16`` holding the bf16 bit pattern (numpy has no bfloat16).
"""

from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

DTYPES = ("tf32", "bf16", "fp16")
FAMILIES = ("dyadic", "normal", "uniform")
STREAM_A, STREAM_B, STREAM_C = 0, 1, 2

_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _seed_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([seed], dtype=np.uint64) * GOLDEN + np.uint64(stream)
        return _mix(s)[0]


def raw_u64(seed: int, stream: int, offset: int, n: int) -> np.ndarray:
    """Draws ``offset .. offset+n-1`` of stream (seed, stream) as uint64."""
    key = _seed_key(seed, stream)
    out = np.empty(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for lo in range(0, n, _CHUNK):
            hi = min(n, lo + _CHUNK)
            ctr = np.arange(offset + lo + 1, offset + hi + 1, dtype=np.uint64)
            out[lo:hi] = _mix(key + ctr * GOLDEN)
    return out


def uniform01(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """n uniform doubles in [0, 1), each exactly k * 2**-53."""
    r = raw_u64(seed, stream, offset, n)
    return (r >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _normal64(seed: int, stream: int, n: int) -> np.ndarray:
    """n N(0,1) doubles by Box-Muller; pair p uses draws 2p and 2p+1."""
    pairs = (n + 1) // 2
    out = np.empty(2 * pairs, dtype=np.float64)
    for lo in range(0, pairs, _CHUNK):
        hi = min(pairs, lo + _CHUNK)
        u = uniform01(seed, stream, 2 * (hi - lo), offset=2 * lo)
        u1 = 1.0 - u[0::2]          # (0, 1]: log is finite
        u2 = u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        t = 2.0 * np.pi * u2
        out[2 * lo:2 * hi:2] = r * np.cos(t)
        out[2 * lo + 1:2 * hi:2] = r * np.sin(t)
    return out[:n]


def _values64(family: str, seed: int, stream: int, n: int) -> np.ndarray:
    if family == "dyadic":
        return np.floor(9.0 * uniform01(seed, stream, n)) - 4.0
    if family == "normal":
        return _normal64(seed, stream, n)
    if family == "uniform":
        return 2.0 * uniform01(seed, stream, n) - 1.0
    raise ValueError(f"unknown family {family!r}")


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits.

    NaN is not produced by any family, so it needs no special case here.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def store(v64: np.ndarray, dtype: str) -> np.ndarray:
    """Round doubles to the storage type of ``dtype`` (via fp32, RNE each step)."""
    f32 = v64.astype(np.float32)
    if dtype == "tf32":
        return f32
    if dtype == "bf16":
        return f32_to_bf16_bits(f32)
    if dtype == "fp16":
        return f32.astype(np.float16)
    raise ValueError(f"unknown dtype {dtype!r}")


def matrix(family: str, dtype: str, rows: int, cols: int, seed: int, stream: int) -> np.ndarray:
    """One row-major ``rows x cols`` operand in the storage type of ``dtype``."""
    v = _values64(family, seed, stream, rows * cols)
    return store(v, dtype).reshape(rows, cols)


def c_matrix(family: str, rows: int, cols: int, seed: int) -> np.ndarray:
    """The initial C (always fp32), drawn from stream 2."""
    v = _values64(family, seed, STREAM_C, rows * cols)
    return v.astype(np.float32).reshape(rows, cols)


def problem(M: int, N: int, K: int, dtype: str, family: str, seed: int,
            c_family: str | None = None):
    """A (M x K), B (K x N) and, if ``c_family`` is given, C0 (M x N fp32)."""
    A = matrix(family, dtype, M, K, seed, STREAM_A)
    B = matrix(family, dtype, K, N, seed, STREAM_B)
    C0 = c_matrix(c_family, M, N, seed) if c_family else None
    return A, B, C0


# The workloads of the deterministic-GEMM study: (name, dtype, (M, N, K),
# family of A and B, alpha, beta, family of C0, seed, gate).
WORKLOADS = [
    ("dyadic256", "tf32", (256, 256, 256), "dyadic", 1.0, 0.0, None, 0, "exact"),
    ("square2048", "tf32", (2048, 2048, 2048), "normal", 1.0, 0.0, None, 1, "rel_rms"),
    ("square4096", "tf32", (4096, 4096, 4096), "normal", 1.0, 0.0, None, 2, "rel_rms"),
    ("square8192", "tf32", (8192, 8192, 8192), "normal", 1.0, 0.0, None, 2, "rel_rms"),
    ("square4096", "bf16", (4096, 4096, 4096), "normal", 1.0, 0.0, None, 3, "rel_rms"),
    ("square8192", "bf16", (8192, 8192, 8192), "normal", 1.0, 0.0, None, 3, "rel_rms"),
    ("square4096", "fp16", (4096, 4096, 4096), "normal", 1.0, 0.0, None, 3, "rel_rms"),
    ("square8192", "fp16", (8192, 8192, 8192), "normal", 1.0, 0.0, None, 3, "rel_rms"),
    # skinny M (few rows against wide, deep operands), where the dispatcher
    # may exchange the operands' roles
    ("skinny16x8192x8192", "bf16", (16, 8192, 8192), "normal", 1.0, 0.0, None, 5, "rel_rms"),
    ("skinny32x16384x4096", "tf32", (32, 16384, 4096), "normal", 1.0, 0.0, None, 5, "rel_rms"),
] + [
    (f"tail{M}x{N}x{K}", dt, (M, N, K), "uniform", 1.5, 0.5, "normal", 4, "rel_rms")
    for dt in ("tf32", "bf16")
    for (M, N, K) in ((768, 768, 768), (8191, 4097, 2049), (16384, 1024, 4096),
                      (128, 8192, 8192), (4096, 4096, 512))
]

# The row-operator workloads: rows x width of the wide-row softmax, RMSNorm
# and LayerNorm cases ("Scale coverage exposes a remaining GEMM gap",
# section "Reductions: wide rows and large working sets"), fp32.
ROWOP_SHAPES = [(37, 8191), (1024, 8192), (1024, 16384), (4096, 8192), (8192, 4096), (16384, 4096)]
ROWOPS = ("softmax", "rmsnorm", "layernorm")


def rowop_inputs(rows: int, width: int, seed: int = 6):
    """X ~ N(0,1) (rows x width), gamma = 1 + U(-1/2, 1/2) and beta ~ N(0, 1/4)
    per column, all fp32. The pages give no distribution; these keep every
    operator's output of order one."""
    x = matrix("normal", "tf32", rows, width, seed, 0)
    gamma = (1.0 + 0.5 * matrix("uniform", "tf32", 1, width, seed, 1)[0].astype(np.float64)).astype(np.float32)
    beta = (0.5 * matrix("normal", "tf32", 1, width, seed, 2)[0].astype(np.float64)).astype(np.float32)
    return x, gamma, beta


# rel_rms bounds per dtype (the deterministic-GEMM acceptance gates).
REL_RMS_BOUND = {"tf32": 1e-3, "bf16": 8e-3, "fp16": 8e-3}
