"""Python face of the FP64 CPU oracles: GEMM (``gemm_oracle.c``) and the
row operators softmax, RMSNorm and LayerNorm (``rowops.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the library
``shape_adaptive_tile_gb300`` never does, and this package never imports the
library. It compiles its C source with the host compiler on first use.

``rel_rms`` follows the accuracy figure of "Measured data point on
fixed-tile vs shape-adaptive GEMM" (section "What we measured"), which the
page reports but never defines; the reading used here is
``sqrt(sum((c - ref)^2)) / sqrt(sum(ref^2))`` over all outputs, in double.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "gemm_oracle.c"), os.path.join(_HERE, "rowops.c")]
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_CODES = {"tf32": 0, "fp32": 0, "bf16": 1, "fp16": 2}
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O3", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so``; returns its path.

    A stale library is deleted before the compiler runs, so a failed build
    never leaves an old one in place.
    """
    os.makedirs(_BUILD, exist_ok=True)
    fresh = os.path.exists(_LIB) and all(os.path.getmtime(_LIB) >= os.path.getmtime(f) for f in _SRCS)
    if fresh and not force:
        return _LIB
    if os.path.exists(_LIB):
        os.remove(_LIB)
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-o", tmp, *_SRCS, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p, d = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
            lib.oracle_gemm_rows.argtypes = [i64, i64, i64, ctypes.c_int, p, p, p, d, d, i64, i64, p, p]
            lib.oracle_gemm_rows.restype = ctypes.c_int
            lib.oracle_gemm_entries.argtypes = [i64, i64, i64, ctypes.c_int, p, p, p, d, d, i64, p, p, p, p]
            lib.oracle_gemm_entries.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [ctypes.c_int, ctypes.c_uint32]
            lib.oracle_decode.restype = ctypes.c_double
            lib.oracle_threads.argtypes = []
            lib.oracle_threads.restype = ctypes.c_int
            lib.oracle_softmax_rows.argtypes = [p, i64, i64, i64, p]
            lib.oracle_softmax_rows.restype = None
            lib.oracle_rmsnorm_rows.argtypes = [p, i64, p, i64, i64, d, p]
            lib.oracle_rmsnorm_rows.restype = None
            lib.oracle_layernorm_rows.argtypes = [p, i64, p, p, i64, i64, d, p]
            lib.oracle_layernorm_rows.restype = None
            _lib = lib
    return _lib


def _code(dtype: str) -> int:
    try:
        return _CODES[dtype]
    except KeyError:
        raise ValueError(f"unknown dtype {dtype!r}") from None


def _operand(x: np.ndarray, dtype: str) -> np.ndarray:
    want = {0: np.float32, 1: np.uint16, 2: np.float16}[_code(dtype)]
    if x.dtype != want:
        raise TypeError(f"{dtype} operand must be stored as {np.dtype(want).name}, got {x.dtype}")
    return np.ascontiguousarray(x)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _prep(A, B, C0, beta, dtype):
    A = _operand(A, dtype)
    B = _operand(B, dtype)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {A.shape} x {B.shape}")
    if beta != 0.0:
        if C0 is None:
            raise ValueError("beta != 0 needs C0")
        C0 = np.ascontiguousarray(C0, dtype=np.float32)
        if C0.shape != (M, N):
            raise ValueError("C0 must be M x N")
    else:
        C0 = None if C0 is None else np.ascontiguousarray(C0, dtype=np.float32)
    return A, B, C0, M, N, K


def gemm(A, B, C0=None, alpha=1.0, beta=0.0, dtype="tf32", row_begin=0, row_end=None):
    """Rows [row_begin, row_end) of alpha*A*B + beta*C0; returns (f64, f32)."""
    A, B, C0, M, N, K = _prep(A, B, C0, beta, dtype)
    row_end = M if row_end is None else row_end
    rows = row_end - row_begin
    out64 = np.empty((rows, N), dtype=np.float64)
    out32 = np.empty((rows, N), dtype=np.float32)
    rc = _load().oracle_gemm_rows(M, N, K, _code(dtype), _ptr(A), _ptr(B), _ptr(C0),
                                  float(alpha), float(beta), row_begin, row_end,
                                  _ptr(out64), _ptr(out32))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_rows failed ({rc})")
    return out64, out32


def _exact_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """The exact values of stored operand elements as doubles: fp32 and fp16
    widen exactly; a bf16 bit pattern is the top half of the fp32 with the
    same sign, exponent and leading fraction bits."""
    code = _code(dtype)
    if code == 1:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def gemm_full(A, B, C0=None, alpha=1.0, beta=0.0, dtype="tf32"):
    """All of alpha*A*B + beta*C0 in double, with numpy's float64 matrix
    product as the sum over k; returns (f64, f32).

    The same definition as :func:`gemm`, with a library matrix product as
    its one step: the operands enter as the exact doubles of their stored
    bits, ``acc = A @ B`` in float64, ``out64 = alpha*acc + beta*C0`` (the
    beta term only when beta != 0), ``out32`` one round to nearest even.
    The library sums over k in its own blocked order, so ``out64`` can differ
    from :func:`gemm`'s ascending-k double sum by a few units in the last
    place of double; where every partial sum is exact in double (the dyadic
    family) both are exact and equal bit for bit. It exists for complete
    outputs of the largest benchmark shapes, where the plain loop streams B
    from memory once per row of A.
    """
    A, B, C0, M, N, K = _prep(A, B, C0, beta, dtype)
    acc = _exact_f64(A, dtype) @ _exact_f64(B, dtype) if K > 0 else np.zeros((M, N))
    out64 = float(alpha) * acc
    del acc
    if beta != 0.0:
        out64 += float(beta) * C0.astype(np.float64)
    return out64, out64.astype(np.float32)


def gemm_entries(A, B, rows, cols, C0=None, alpha=1.0, beta=0.0, dtype="tf32"):
    """Entries (rows[e], cols[e]) of alpha*A*B + beta*C0; returns (f64, f32)."""
    A, B, C0, M, N, K = _prep(A, B, C0, beta, dtype)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols differ in length")
    n = rows.size
    out64 = np.empty(n, dtype=np.float64)
    out32 = np.empty(n, dtype=np.float32)
    rc = _load().oracle_gemm_entries(M, N, K, _code(dtype), _ptr(A), _ptr(B), _ptr(C0),
                                     float(alpha), float(beta), n, _ptr(rows), _ptr(cols),
                                     _ptr(out64), _ptr(out32))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_entries failed ({rc})")
    return out64, out32


def decode(dtype: str, bits: int) -> float:
    """Exact value of one stored element given its bit pattern."""
    return _load().oracle_decode(_code(dtype), int(bits))


def threads() -> int:
    """OpenMP threads the oracle runs on."""
    return _load().oracle_threads()


def rel_rms(c, ref64) -> float:
    """sqrt(sum (c - ref)^2) / sqrt(sum ref^2), accumulated in double."""
    c = np.asarray(c, dtype=np.float64).ravel()
    r = np.asarray(ref64, dtype=np.float64).ravel()
    den = float(np.sqrt(np.dot(r, r)))
    d = c - r
    num = float(np.sqrt(np.dot(d, d)))
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / den


# ---- row operators (rowops.c) ---------------------------------------------------


def _rows_in(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim != 2:
        raise ValueError("x must be rows x width")
    return x


def _vec(v, width):
    if v is None:
        return None
    v = np.ascontiguousarray(v, dtype=np.float32)
    if v.shape != (width,):
        raise ValueError("gamma/beta must have one entry per column")
    return v


def softmax(x):
    """Row-wise softmax of fp32 x (rows x width), in double."""
    x = _rows_in(x)
    y = np.empty(x.shape, np.float64)
    _load().oracle_softmax_rows(_ptr(x), x.shape[1], x.shape[0], x.shape[1], _ptr(y))
    return y


def rmsnorm(x, gamma=None, eps=1e-5):
    """Row-wise RMSNorm of fp32 x with optional per-column gamma, in double."""
    x = _rows_in(x)
    g = _vec(gamma, x.shape[1])
    y = np.empty(x.shape, np.float64)
    _load().oracle_rmsnorm_rows(_ptr(x), x.shape[1], _ptr(g) if g is not None else None, x.shape[0], x.shape[1],
                                float(eps), _ptr(y))
    return y


def layernorm(x, gamma=None, beta=None, eps=1e-5):
    """Row-wise LayerNorm (biased variance) of fp32 x with optional gamma and beta, in double."""
    x = _rows_in(x)
    g, b = _vec(gamma, x.shape[1]), _vec(beta, x.shape[1])
    y = np.empty(x.shape, np.float64)
    _load().oracle_layernorm_rows(_ptr(x), x.shape[1], _ptr(g) if g is not None else None,
                                  _ptr(b) if b is not None else None, x.shape[0], x.shape[1], float(eps), _ptr(y))
    return y
