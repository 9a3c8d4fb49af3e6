"""Acceptance checks shared by the GPU parity tests.

The gates are those of the deterministic-GEMM study: bit-exact equality
with the fp32-rounded oracle where the exact result is representable (the
dyadic family), else rel_rms against the FP64 oracle within the dtype's
bound, plus identical bits over repeated runs.
"""
import numpy as np

import oracle


def bit_exact_mismatches(got, ref32) -> int:
    """Number of elements whose fp32 bits differ (NaN never equals)."""
    g = np.ascontiguousarray(got, dtype=np.float32).view(np.uint32)
    r = np.ascontiguousarray(ref32, dtype=np.float32).view(np.uint32)
    if g.shape != r.shape:
        raise ValueError(f"shape {g.shape} != {r.shape}")
    bad = g != r
    bad |= np.isnan(np.asarray(got, dtype=np.float32))
    return int(np.count_nonzero(bad))


def assert_bit_exact(got, ref32, what=""):
    n = bit_exact_mismatches(got, ref32)
    assert n == 0, f"{what}: {n} of {np.size(ref32)} outputs differ from the oracle's fp32 bits"


def assert_rel_rms(got, ref64, bound, what=""):
    got = np.asarray(got)
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    r = oracle.rel_rms(got, ref64)
    assert r <= bound, f"{what}: rel_rms {r:.3e} > {bound:.1e}"
    return r
