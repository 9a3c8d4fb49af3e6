"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports
every function include/gemm.h and include/rowops.h declare, fails cleanly
when no device is present, and its dispatcher (host logic only) makes sane
choices."""
import ctypes
import os
import re

import pytest

import shape_adaptive_tile_gb300 as sat

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADERS = [os.path.join(INCLUDE, "gemm.h"), os.path.join(INCLUDE, "rowops.h")]  # the C ABI
# (include/gemm_device.cuh is the device routine's CUDA C++ header; the library
# builds it into gemm_selftest_device_call.)


@pytest.fixture(scope="module")
def lib():
    sat.build()
    return sat.lib()


def _declared():
    text = "".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:gemm|rowop)_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for fn in ("gemm_plan_create", "gemm_run", "gemm_plan_destroy", "gemm_last_error", "gemm_plan_describe",
               "rowop_softmax", "rowop_rmsnorm", "rowop_layernorm"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared()
    assert set(names) == set(sat.EXPORTS)
    for fn in names:
        assert hasattr(lib, fn), fn
        assert ctypes.cast(getattr(lib, fn), ctypes.c_void_p).value


def test_null_plan_and_destroy_are_safe_without_a_device(lib):
    assert sat.gemm_run(None, 0, 0, 0, 1.0, 0.0, None) == -1
    sat.gemm_plan_destroy(None)
    assert sat.gemm_plan_describe(None) == ""


def test_plan_create_fails_cleanly_without_a_gpu(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(sat.GemmError):
        sat.gemm_plan_create(128, 128, 128, "tf32")
    assert sat.gemm_last_error()


def _choice(M, N, K, dt, sms=152, tma=True):
    bn, cg, raster, group, splits, cload, sk, swap, stages, source = \
        sat.gemm_select_config(M, N, K, dt, sms, tma).split(",")
    return int(bn), int(cg), int(raster), int(group), int(splits), source


def _swap(M, N, K, dt, tma=True):
    return int(sat.gemm_select_config(M, N, K, dt, 152, tma).split(",")[7])


@pytest.mark.parametrize("dt", ["tf32", "bf16", "fp16"])
def test_dispatcher_choices_are_compiled_variants(dt):
    for M, N, K in [(256, 256, 256), (2048, 2048, 2048), (8192, 8192, 8192), (768, 768, 768),
                    (8191, 4097, 2049), (16384, 1024, 4096), (128, 8192, 8192), (4096, 4096, 512), (1, 1, 1),
                    (16, 8192, 8192), (64, 4096, 520)]:
        for tma in (True, False):
            bn, cg, raster, group, splits, _ = _choice(M, N, K, dt, tma=tma)
            swap = _swap(M, N, K, dt, tma)
            assert cg in (1, 2) and raster in (0, 1) and group >= 1
            assert 1 <= splits <= 16
            if swap:   # swapped variants: 1-SM, 32/64/128 rows of C per tile
                assert tma and cg == 1 and bn in (32, 64, 128)
            else:
                assert bn in (64, 128, 256)
            if not tma:   # class-view kernels: 1-SM 128 or 256 columns, CTA-pair 256
                assert (cg, bn) in ((1, 128), (1, 256), (2, 256)) and swap == 0


def test_dispatcher_swaps_operands_for_skinny_m_only():
    assert _swap(1, 4096, 4096, "tf32") == 1 and _choice(1, 4096, 4096, "tf32")[0] == 32
    assert _swap(32, 4096, 4096, "bf16") == 1 and _choice(32, 4096, 4096, "bf16")[0] == 32
    assert _swap(48, 4096, 4096, "bf16") == 0
    assert _swap(16, 4100, 4096, "bf16", tma=False) == 0   # no TMA, no swapped variant


def test_dispatcher_fills_the_machine_for_skinny_m():
    # 128 x 8192: one 128x256 tile per SM would occupy 32 of 152 SMs; the
    # choice must engage at least half of them.
    for dt in ("tf32", "bf16"):
        bn, cg, _, _, splits, _ = _choice(128, 8192, 8192, dt)
        tiles = -(-128 // (128 * cg)) * -(-8192 // bn) * splits
        assert min(tiles * cg, 152) >= 76


def test_dispatcher_splits_k_only_when_tiles_leave_sms_idle():
    # A long K over few tiles: the rule splits K; a large square problem never.
    assert _choice(256, 256, 16384, "bf16")[4] > 1
    assert _choice(4096, 4096, 4096, "bf16")[4] == 1
    assert _choice(8192, 8192, 8192, "tf32")[4] == 1


def _cload(M, N, K, dt):
    return int(sat.gemm_select_config(M, N, K, dt, 152, True).split(",")[5])


def test_dispatcher_takes_c_through_the_ring_only_for_short_k():
    # beta != 0: the ring measured faster where C is a large share of a tile's
    # traffic (few k-blocks), slower behind a long K loop. Rule and table agree.
    assert _cload(3000, 3000, 256, "bf16") == 0      # rule, 4 k-blocks
    assert _cload(3000, 3000, 8192, "bf16") == 1     # rule, 128 k-blocks
    assert _cload(3000, 3000, 1024, "tf32") == 0     # rule, 32 k-blocks
    assert _cload(3000, 3000, 1056, "tf32") == 1     # rule, 33 k-blocks
    assert _cload(4096, 4096, 512, "bf16") == 0      # table
    # table: the long-K shape loads C in the epilogue (stream-K runs do too)
    for dt in ("bf16", "tf32"):
        f = sat.gemm_select_config(16384, 1024, 4096, dt, 152, True).split(",")
        assert f[5] == "1" or f[6] == "1"


def _sk(M, N, K, dt, sms=152):
    return int(sat.gemm_select_config(M, N, K, dt, sms, True).split(",")[6])


def test_dispatcher_stream_k_only_past_one_wave_with_a_partial_last_one():
    assert _sk(6144, 6144, 4096, "bf16") == 1    # 576 pair tiles: 7 waves of 76 plus 44
    assert _sk(5000, 5000, 5000, "tf32") == 1
    assert _sk(2000, 2000, 4096, "bf16") == 0    # 64 pair tiles: less than one wave
    assert _sk(4864, 19456, 4096, "bf16") == 0   # 19 x 76 pair tiles: whole waves
    assert _sk(3000, 3000, 128, "bf16") == 0     # K too short for the fix-up to pay


def test_dispatcher_rejects_bad_arguments():
    with pytest.raises(sat.GemmError):
        sat.gemm_select_config(-1, 4, 4, "tf32", 152, True)
    with pytest.raises(sat.GemmError):
        sat.gemm_select_config(4, 4, 4, "tf32", 0, True)


def test_gemm_source_hash_ignores_only_the_row_operators(tmp_path, monkeypatch):
    # The recorded GEMM traffic is keyed on this hash: editing a row-operator
    # file must leave it alone, editing a GEMM source must change it.
    import importlib
    b = importlib.import_module("shape_adaptive_tile_gb300.build")
    src = tmp_path / "csrc"
    inc = tmp_path / "include"
    src.mkdir()
    inc.mkdir()
    for name in ("gemm_kernel.cuh", "rowops.cu", "api.cu"):
        (src / name).write_text(name)
    for name in ("gemm.h", "rowops.h"):
        (inc / name).write_text(name)
    monkeypatch.setattr(b, "CSRC", str(src))
    monkeypatch.setattr(b, "INCLUDE", str(inc))
    h0, f0 = b.gemm_source_hash(), b.source_hash()
    (src / "rowops.cu").write_text("changed")
    (inc / "rowops.h").write_text("changed")
    assert b.gemm_source_hash() == h0 and b.source_hash() != f0
    (src / "gemm_kernel.cuh").write_text("changed")
    assert b.gemm_source_hash() != h0


def test_source_hash_ignores_comments_and_layout_only(tmp_path, monkeypatch):
    # A profile stays valid across a comment edit, not across a code edit,
    # and a comment marker inside a string literal is code.
    import importlib
    b = importlib.import_module("shape_adaptive_tile_gb300.build")
    src = tmp_path / "csrc"
    inc = tmp_path / "include"
    src.mkdir()
    inc.mkdir()
    (inc / "gemm.h").write_text("int f(int);\n")
    k = src / "gemm_kernel.cuh"
    k.write_text('int f(int x) { return x + 1; }  // one\nconst char* s = "a//b";\n')
    monkeypatch.setattr(b, "CSRC", str(src))
    monkeypatch.setattr(b, "INCLUDE", str(inc))
    h0 = b.gemm_source_hash()
    k.write_text('/* new\n   block */ int f(int x)\n{\n  return x + 1;  // two\n}\nconst char* s = "a//b";\n')
    assert b.gemm_source_hash() == h0
    k.write_text('int f(int x) { return x + 2; }  // one\nconst char* s = "a//b";\n')
    assert b.gemm_source_hash() != h0
    k.write_text('int f(int x) { return x + 1; }  // one\nconst char* s = "a//c";\n')
    assert b.gemm_source_hash() != h0
    k.write_text("int f(int x) { return x + 1; }\nconst char* s = \"a//b\"; char c = '/';\n")
    assert b.gemm_source_hash() != h0


def test_noalloc_scratch_holds_every_dispatcher_choice_on_a_gb300():
    # gemm_run_noalloc keeps its partial tiles in a fixed array of 32 MiB
    # minus a 4 KiB status area (status word, then one stream-K counter per
    # CTA from byte 256). On a 152-SM GB300 every choice of the dispatcher
    # must fit, from skinny to square, short K to long: its K splits and
    # stream-K grids keep the partial tiles within one 128 x 256 float tile
    # per SM.
    sms, limit, counters = 152, (32 << 20) - 4096, (4096 - 256) // 4
    worst = 0
    for dt in ("tf32", "bf16", "fp16"):
        for M in (1, 16, 32, 100, 128, 129, 256, 300, 1000, 2048, 4096, 8191, 16384, 65536):
            for N in (8, 256, 1000, 4096, 8192, 19456, 65536):
                for K in (64, 512, 2049, 8192, 65536):
                    f = sat.gemm_select_config(M, N, K, dt, sms, True).split(",")
                    bn, cg, splits, sk = int(f[0]), int(f[1]), int(f[4]), int(f[6])
                    rows = 128 * cg
                    need = splits * (-(-M // rows) * rows) * N * 4 if splits > 1 else 0
                    if sk:
                        need = max(need, (sms // cg) * cg * 128 * bn * 4)
                        assert (sms // cg) * cg <= counters
                    worst = max(worst, need)
                    assert need <= limit, (dt, M, N, K, f, need)
    assert 0 < worst <= sms * 128 * 256 * 4


def _fields(M, N, K, dt, tma=True):
    return sat.gemm_select_config(M, N, K, dt, 152, tma).split(",")


def test_dispatcher_reports_the_ring_depth():
    # The chosen kernel's shared-memory ring: 6 stages for the CTA-pair
    # 256-wide tile, 4 for the 1-SM 256-wide tile, 8 for 1-SM 64-wide ones.
    f = _fields(8192, 8192, 8192, "tf32")
    assert f[:2] == ["256", "2"] and f[8] == "6" and f[9] == "table"
    f = _fields(768, 768, 768, "tf32")
    assert f[0] == "64" and f[8] == "8"
    for M, N, K in [(5000, 5000, 5000), (333, 517, 389), (1, 4096, 4096)]:
        for dt in ("tf32", "bf16"):
            assert int(_fields(M, N, K, dt)[8]) >= 2


def test_dispatcher_bucket_serves_shapes_next_to_the_table():
    # One row or one k off a swept shape: the same power-of-two bucket, the
    # swept shape's choice.
    for M, N, K, dt, near in [(8192, 8192, 8191, "bf16", (8192, 8192, 8192)),
                              (8000, 8100, 8192, "tf32", (8192, 8192, 8192)),
                              (4095, 4096, 4096, "bf16", (4096, 4096, 4096)),
                              (16000, 1000, 4000, "tf32", (16384, 1024, 4096)),
                              (120, 8192, 8000, "bf16", (128, 8192, 8192))]:
        f, g = _fields(M, N, K, dt), _fields(*near, dt)
        assert f[9] == "bucket" and g[9] == "table", (M, N, K, f, g)
        assert f[:9] == g[:9], (M, N, K, f, g)
    # Outside every bucket: the rule.
    assert _fields(1500, 1500, 1500, "bf16")[9] == "rule"
    # The misaligned (8191, 4097, 2049) row serves plain-load shapes only.
    assert _fields(8190, 4099, 2051, "tf32", tma=False)[9] == "bucket"
    assert _fields(8192, 8192, 4096, "tf32")[9] != "bucket" or _fields(8192, 8192, 4096, "tf32")[1] == "2"


def test_rule_picks_the_raster_group_with_least_modelled_traffic():
    # No table row near either shape, 76 CTA pairs. bf16 12288^3: a wave of
    # 76 tiles spans ~17 operand panels of 6 MB at best (groups of 8 or 16
    # tile-rows), more than L2 keeps between waves, so the group must keep a
    # wave square; groups of 1 would touch ~50 panels per wave.
    f = _fields(12288, 12288, 12288, "bf16")
    assert f[9] == "rule" and f[1] == "2" and int(f[3]) >= 8
    # bf16 6144 x 6144 x 4096: B's 24 column panels (48 MB) fit in L2, so
    # waves running along whole tile-rows (group 1) read A and B once.
    f = _fields(6144, 6144, 4096, "bf16")
    assert f[9] == "rule" and f[2:4] == ["0", "1"]
