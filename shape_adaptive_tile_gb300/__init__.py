"""Deterministic, shape-adaptive dense GEMM for GB300 (sm_103a).

A thin ctypes binding over the C ABI of ``include/gemm.h``: the functions
below have the C names and only marshal arguments; every step of the GEMM
runs in the library's CUDA kernels. Operand pointers are plain integers
(for example ``torch.Tensor.data_ptr()``); streams are ``cudaStream_t``
values (for example ``torch.cuda.current_stream().cuda_stream``).

Nothing here falls back to another implementation: if the library is not
built, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB, build  # noqa: F401  (build is part of the public surface)

GEMM_TF32, GEMM_BF16, GEMM_FP16 = 0, 1, 2
DTYPES = {"tf32": GEMM_TF32, "bf16": GEMM_BF16, "fp16": GEMM_FP16}
STATUS = {0: "GEMM_OK", -1: "GEMM_ERR_ARG", -2: "GEMM_ERR_ARCH", -3: "GEMM_ERR_ALIGN",
          -4: "GEMM_ERR_LAUNCH", -5: "GEMM_ERR_TIMEOUT", -6: "GEMM_ERR_NOMEM"}

# Every function the C ABI exports (include/gemm.h).
EXPORTS = ("gemm_plan_create", "gemm_plan_create_config", "gemm_plan_create_ex", "gemm_run", "gemm_run_ex",
           "gemm_run_host", "gemm_plan_destroy", "gemm_plan_status", "gemm_plan_describe", "gemm_last_error",
           "gemm_selftest_bounded_wait", "gemm_select_config", "gemm_run_noalloc", "gemm_selftest_device_call",
           "gemm_device_prepare",
           "rowop_softmax", "rowop_rmsnorm", "rowop_layernorm")

_lock = threading.Lock()
_lib = None


class GemmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError(f"CUDA library not built ({LIB}); run shape_adaptive_tile_gb300.build()")
            L = ctypes.CDLL(LIB)
            i64, vp, f32, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
            L.gemm_plan_create.argtypes = [i64, i64, i64, i32]
            L.gemm_plan_create.restype = vp
            L.gemm_plan_create_config.argtypes = [i64, i64, i64, i32, ctypes.c_char_p]
            L.gemm_plan_create_config.restype = vp
            L.gemm_run.argtypes = [vp, vp, vp, vp, f32, f32, vp]
            L.gemm_run.restype = i32
            L.gemm_plan_create_ex.argtypes = [i64, i64, i64, i32, i32, i32, i32, ctypes.c_char_p]
            L.gemm_plan_create_ex.restype = vp
            L.gemm_run_ex.argtypes = [vp, vp, i64, vp, i64, vp, i64, f32, f32, vp]
            L.gemm_run_ex.restype = i32
            L.gemm_run_host.argtypes = [vp, vp, vp, vp, f32, f32, vp, vp, vp, vp]
            L.gemm_run_host.restype = i32
            L.gemm_plan_destroy.argtypes = [vp]
            L.gemm_plan_destroy.restype = None
            L.gemm_plan_status.argtypes = [vp]
            L.gemm_plan_status.restype = i32
            L.gemm_plan_describe.argtypes = [vp]
            L.gemm_plan_describe.restype = ctypes.c_char_p
            L.gemm_last_error.argtypes = []
            L.gemm_last_error.restype = ctypes.c_char_p
            L.gemm_selftest_bounded_wait.argtypes = [ctypes.c_uint64]
            L.gemm_selftest_bounded_wait.restype = i32
            L.gemm_run_noalloc.argtypes = [i64, i64, i64, i32, vp, vp, vp, f32, f32, vp]
            L.gemm_selftest_device_call.argtypes = [i64, i64, i64, i32, vp, vp, vp, f32, f32, i32, vp]
            L.gemm_selftest_device_call.restype = i32
            L.gemm_device_prepare.argtypes = [i64, i64, i64, i32, vp, vp, vp, f32, f32, i32, vp, i64]
            L.gemm_device_prepare.restype = i32
            L.rowop_softmax.argtypes = [vp, i64, vp, i64, i64, i64, vp]
            L.rowop_softmax.restype = i32
            L.rowop_rmsnorm.argtypes = [vp, i64, vp, vp, i64, i64, i64, f32, vp]
            L.rowop_rmsnorm.restype = i32
            L.rowop_layernorm.argtypes = [vp, i64, vp, vp, vp, i64, i64, i64, f32, vp]
            L.rowop_layernorm.restype = i32
            L.gemm_run_noalloc.restype = i32
            L.gemm_select_config.argtypes = [i64, i64, i64, i32, i32, i32, ctypes.c_char_p, i32]
            L.gemm_select_config.restype = i32
            _lib = L
    return _lib


def _dt(dtype) -> int:
    return DTYPES[dtype] if isinstance(dtype, str) else int(dtype)


def _p(x) -> int | None:
    if x is None:
        return None
    return int(x.data_ptr()) if hasattr(x, "data_ptr") else int(x)


def gemm_last_error() -> str:
    return lib().gemm_last_error().decode()


def gemm_plan_create(M: int, N: int, K: int, dtype) -> int:
    h = lib().gemm_plan_create(M, N, K, _dt(dtype))
    if not h:
        raise GemmError(-1, gemm_last_error())
    return h


def gemm_plan_create_config(M: int, N: int, K: int, dtype, config: str | None) -> int:
    h = lib().gemm_plan_create_config(M, N, K, _dt(dtype), config.encode() if config else None)
    if not h:
        raise GemmError(-1, gemm_last_error())
    return h


C_TYPES = {"fp32": 0, "bf16": 1, "fp16": 2}


def gemm_plan_create_ex(M: int, N: int, K: int, dtype, trans_a: bool, trans_b: bool, c_type="fp32",
                        config: str | None = None) -> int:
    h = lib().gemm_plan_create_ex(M, N, K, _dt(dtype), int(bool(trans_a)), int(bool(trans_b)),
                                  C_TYPES[c_type] if isinstance(c_type, str) else int(c_type),
                                  config.encode() if config else None)
    if not h:
        raise GemmError(-1, gemm_last_error())
    return h


def gemm_run(plan: int, A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None) -> int:
    return lib().gemm_run(plan, _p(A), _p(B), _p(C), alpha, beta, _p(stream))


def gemm_run_ex(plan: int, A, lda: int, B, ldb: int, C, ldc: int, alpha: float = 1.0, beta: float = 0.0,
                stream=None) -> int:
    return lib().gemm_run_ex(plan, _p(A), lda, _p(B), ldb, _p(C), ldc, alpha, beta, _p(stream))


def gemm_run_host(plan: int, hA, hB, hC, alpha, beta, dA, dB, dC, stream=None) -> int:
    return lib().gemm_run_host(plan, _p(hA), _p(hB), _p(hC), alpha, beta, _p(dA), _p(dB), _p(dC), _p(stream))


def gemm_run_noalloc(M: int, N: int, K: int, dtype, A, B, C, alpha: float = 1.0, beta: float = 0.0,
                     stream=None) -> int:
    """The allocation-free GEMM (see include/gemm.h): no plan, fixed scratch."""
    return lib().gemm_run_noalloc(M, N, K, _dt(dtype), _p(A), _p(B), _p(C), alpha, beta, _p(stream))


def gemm_selftest_device_call(M: int, N: int, K: int, dtype, A, B, C, alpha: float = 1.0, beta: float = 0.0,
                              cta_group: int = 1, stream=None) -> int:
    """GEMM then ReLU in one launch, the GEMM being the device-callable routine (see include/gemm.h)."""
    return lib().gemm_selftest_device_call(M, N, K, _dt(dtype), _p(A), _p(B), _p(C), alpha, beta, cta_group,
                                           _p(stream))


def gemm_device_prepare(M: int, N: int, K: int, dtype, A, B, C, alpha: float, beta: float, cta_group: int,
                        params, params_bytes: int) -> int:
    """Fill the device routine's launch parameters into host memory `params` (see include/gemm.h)."""
    return lib().gemm_device_prepare(M, N, K, _dt(dtype), _p(A), _p(B), _p(C), alpha, beta, cta_group, _p(params),
                                     params_bytes)


# ---- row operators (include/rowops.h) -----------------------------------------


def rowop_softmax(X, ldx: int, Y, ldy: int, rows: int, width: int, stream=None) -> int:
    return lib().rowop_softmax(_p(X), ldx, _p(Y), ldy, rows, width, _p(stream))


def rowop_rmsnorm(X, ldx: int, gamma, Y, ldy: int, rows: int, width: int, eps: float = 1e-5, stream=None) -> int:
    return lib().rowop_rmsnorm(_p(X), ldx, _p(gamma), _p(Y), ldy, rows, width, eps, _p(stream))


def rowop_layernorm(X, ldx: int, gamma, beta, Y, ldy: int, rows: int, width: int, eps: float = 1e-5,
                    stream=None) -> int:
    return lib().rowop_layernorm(_p(X), ldx, _p(gamma), _p(beta), _p(Y), ldy, rows, width, eps, _p(stream))


def gemm_plan_destroy(plan: int) -> None:
    lib().gemm_plan_destroy(plan)


def gemm_plan_status(plan: int) -> int:
    return lib().gemm_plan_status(plan)


def gemm_plan_describe(plan: int) -> str:
    return lib().gemm_plan_describe(plan).decode()


def gemm_selftest_bounded_wait(timeout_ns: int) -> int:
    return lib().gemm_selftest_bounded_wait(timeout_ns)


def gemm_select_config(M: int, N: int, K: int, dtype, sm_count: int, tma_ok: bool) -> str:
    buf = ctypes.create_string_buffer(64)
    check(lib().gemm_select_config(M, N, K, _dt(dtype), sm_count, int(bool(tma_ok)), buf, 64))
    return buf.value.decode()


def check(status: int) -> None:
    """Raise GemmError for a non-zero status."""
    if status != 0:
        raise GemmError(status, gemm_last_error())


class Plan:
    """Owns one gemm_plan; ``run`` takes device tensors (or raw pointers)."""

    def __init__(self, M: int, N: int, K: int, dtype, config: str | None = None, trans_a: bool = False,
                 trans_b: bool = False, c_type="fp32"):
        self.M, self.N, self.K, self.dtype = M, N, K, dtype
        self.trans_a, self.trans_b = trans_a, trans_b
        if trans_a or trans_b or c_type not in ("fp32", 0):
            self.handle = gemm_plan_create_ex(M, N, K, dtype, trans_a, trans_b, c_type, config)
        else:
            self.handle = gemm_plan_create_config(M, N, K, dtype, config)

    def run(self, A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None, lda: int | None = None,
            ldb: int | None = None, ldc: int | None = None) -> None:
        """C = alpha * op(A) * op(B) + beta * C; the leading dimensions
        default to the dense ones."""
        if lda is None and ldb is None and ldc is None:
            check(gemm_run(self.handle, A, B, C, alpha, beta, stream))
            return
        lda = lda if lda is not None else (self.M if self.trans_a else self.K)
        ldb = ldb if ldb is not None else (self.K if self.trans_b else self.N)
        ldc = ldc if ldc is not None else self.N
        check(gemm_run_ex(self.handle, A, lda, B, ldb, C, ldc, alpha, beta, stream))

    def status(self) -> int:
        return gemm_plan_status(self.handle)

    def describe(self) -> str:
        return gemm_plan_describe(self.handle)

    def close(self) -> None:
        if self.handle:
            gemm_plan_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
