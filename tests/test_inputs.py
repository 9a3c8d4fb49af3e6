"""The seeded input generators: published SplitMix64 values, family ranges,
exact representability, and byte hashes of the exactly-computed families."""
import hashlib
import os

import numpy as np
import pytest

import synth_inputs as si

HASHES = os.path.join(os.path.dirname(__file__), "golden", "input_hashes.txt")


def test_splitmix64_published_seed0_sequence():
    # SplitMix64 (Steele, Lea, Flood 2014) seeded with 0: first four outputs.
    with np.errstate(over="ignore"):
        got = si._mix(np.arange(1, 5, dtype=np.uint64) * si.GOLDEN)
    assert [int(v) for v in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                     0x06C45D188009454F, 0xF88BB8A8724C81EC]


def test_uniform_is_exact_53_bit_grid_and_offsets_compose():
    u = si.uniform01(7, 1, 1000)
    assert np.all((u >= 0) & (u < 1))
    assert np.array_equal(u * 2.0 ** 53, np.floor(u * 2.0 ** 53))
    assert np.array_equal(si.uniform01(7, 1, 400, offset=600), u[600:])


@pytest.mark.parametrize("dtype", ["tf32", "bf16", "fp16"])
def test_dyadic_family_is_integers_minus4_to_4(dtype):
    A = si.matrix("dyadic", dtype, 64, 128, 0, 0)
    v = si.bf16_bits_to_f32(A) if dtype == "bf16" else A.astype(np.float32)
    assert set(np.unique(v).tolist()) == set(range(-4, 5))


def test_normal_and_uniform_moments():
    z = si.matrix("normal", "tf32", 512, 512, 1, 0).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    u = si.matrix("uniform", "tf32", 512, 512, 4, 0).astype(np.float64)
    assert u.min() >= -1.0 and u.max() < 1.0 and abs(u.var() - 1.0 / 3.0) < 0.01


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -20, -2.5], np.float32)
    got = si.bf16_bits_to_f32(si.f32_to_bf16_bits(x))
    assert got.tolist() == [1.0, 1.0 + 2.0 ** -6, 1.0 + 2.0 ** -7, -2.5]


def test_streams_differ_and_seeds_reproduce():
    A1, B1, C1 = si.problem(8, 8, 8, "tf32", "normal", 3, "normal")
    A2, B2, C2 = si.problem(8, 8, 8, "tf32", "normal", 3, "normal")
    assert np.array_equal(A1, A2) and np.array_equal(B1, B2) and np.array_equal(C1, C2)
    assert not np.array_equal(A1, B1)


def _hash_lines():
    out = {}
    with open(HASHES) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, h = line.split()
                out[key] = h
    return out


@pytest.mark.parametrize("key", sorted(_hash_lines()))
def test_input_bytes_match_committed_hashes(key):
    family, dtype, shape, seed, stream = key.split(":")
    r, c = (int(x) for x in shape.split("x"))
    if stream == "C":
        m = si.c_matrix(family, r, c, int(seed))
    else:
        m = si.matrix(family, dtype, r, c, int(seed), int(stream))
    assert hashlib.sha256(m.tobytes()).hexdigest() == _hash_lines()[key]
