"""GPU parity of the row operators (softmax, RMSNorm, LayerNorm) against the
FP64 oracle, through the C ABI, at every rows x width the pages time.

Tolerances follow from fp32 arithmetic: each output is a handful of
rounded operations (exp to 2 ulp, one division or square root) on top of a
sum of at most 32 terms per thread and a 9-level tree across threads, so
its relative error stays below about 3e-6 for N(0,1) rows. The gates are:
softmax max |y - ref| / ref <= 1e-5; the norms max |y - ref| / (|ref| + 1)
<= 1e-5. Every output of every shape is compared, the largest included.
Two runs give the same bits.
"""
import numpy as np
import pytest
import torch

import oracle
import shape_adaptive_tile_gb300 as sat
import synth_inputs as si
from tests.gpu_util import stream

pytestmark = pytest.mark.gpu

TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    sat.build()
    sat.lib()


_cache = {}


def _inputs(rows, width):
    if (rows, width) not in _cache:
        _cache.clear()
        _cache[(rows, width)] = si.rowop_inputs(rows, width)
    return _cache[(rows, width)]


def _device_run(op, x, g, b, ldx=None, ldy=None, y=None):
    rows, width = x.shape[0], x.shape[1] if ldx is None else x.shape[1]
    dx = x if isinstance(x, torch.Tensor) else torch.from_numpy(x).cuda()
    dy = torch.empty_like(dx) if y is None else y
    ldx = dx.shape[1] if ldx is None else ldx
    ldy = dy.shape[1] if ldy is None else ldy
    width = dx.shape[1] if width is None else width
    dg = torch.from_numpy(g).cuda() if g is not None else None
    db = torch.from_numpy(b).cuda() if b is not None else None
    if op == "softmax":
        rc = sat.rowop_softmax(dx, ldx, dy, ldy, rows, width, stream())
    elif op == "rmsnorm":
        rc = sat.rowop_rmsnorm(dx, ldx, dg, dy, ldy, rows, width, 1e-5, stream())
    else:
        rc = sat.rowop_layernorm(dx, ldx, dg, db, dy, ldy, rows, width, 1e-5, stream())
    assert rc == 0, sat.gemm_last_error()
    torch.cuda.synchronize()
    return dy


def _reference(op, x, g, b):
    if op == "softmax":
        return oracle.softmax(x)
    if op == "rmsnorm":
        return oracle.rmsnorm(x, g)
    return oracle.layernorm(x, g, b)


def _check(op, got, ref, what):
    got = got.astype(np.float64)
    err = np.abs(got - ref) / (ref if op == "softmax" else np.abs(ref) + 1.0)
    assert np.all(np.isfinite(got)), what
    worst = float(err.max())
    assert worst <= TOL, f"{what}: max relative error {worst:.3g} > {TOL}"


@pytest.mark.parametrize("rows,width", si.ROWOP_SHAPES)
@pytest.mark.parametrize("op", si.ROWOPS)
def test_rowop_matches_oracle_and_repeats(op, rows, width):
    x, g, b = _inputs(rows, width)
    y1 = _device_run(op, x, g, b)
    y2 = _device_run(op, x, g, b)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32)), "two runs differ"
    _check(op, y1.cpu().numpy(), _reference(op, x, g, b), f"{op} {rows}x{width}")


@pytest.mark.parametrize("op", si.ROWOPS)
@pytest.mark.parametrize("width", [1, 3, 4, 8, 260, 508, 513, 516, 1020, 2048, 2052, 3000, 4100, 6000, 8188, 16385,
                                   32768])
def test_rowop_widths_and_tails(op, width):
    x, g, b = si.rowop_inputs(5, width, seed=7)
    got = _device_run(op, x, g, b).cpu().numpy()
    _check(op, got, _reference(op, x, g, b), f"{op} width {width}")


@pytest.mark.parametrize("op", si.ROWOPS)
@pytest.mark.parametrize("width,ldx,ldy", [(1000, 1100, 1024), (3000, 3100, 3072), (6000, 6004, 6144)])
def test_rowop_strided_and_in_place(op, width, ldx, ldy):
    rows = 9
    x, g, b = si.rowop_inputs(rows, width, seed=8)
    ref = _reference(op, x, g, b)
    # strided: rows ldx apart in X, ldy apart in Y; padding must stay untouched
    xs = np.full((rows, ldx), np.nan, np.float32)
    xs[:, :width] = x
    ys = torch.full((rows, ldy), -7.0, device="cuda")
    dx = torch.from_numpy(xs).cuda()
    if op == "softmax":
        rc = sat.rowop_softmax(dx, ldx, ys, ldy, rows, width, stream())
    elif op == "rmsnorm":
        rc = sat.rowop_rmsnorm(dx, ldx, torch.from_numpy(g).cuda(), ys, ldy, rows, width, 1e-5, stream())
    else:
        rc = sat.rowop_layernorm(dx, ldx, torch.from_numpy(g).cuda(), torch.from_numpy(b).cuda(), ys, ldy, rows,
                                 width, 1e-5, stream())
    assert rc == 0, sat.gemm_last_error()
    torch.cuda.synchronize()
    out = ys.cpu().numpy()
    assert np.all(out[:, width:] == -7.0)
    _check(op, out[:, :width], ref, f"{op} strided")
    # in place
    d = torch.from_numpy(x.copy()).cuda()
    _device_run(op, d, g, b, y=d)
    _check(op, d.cpu().numpy(), ref, f"{op} in place")


def test_rowop_special_values_and_errors():
    # softmax of one column is 1; LayerNorm of one column is beta; RMSNorm without gamma
    x = np.array([[3.0], [-2.0]], np.float32)
    assert np.all(_device_run("softmax", x, None, None).cpu().numpy() == 1.0)
    b = np.array([0.25], np.float32)
    assert np.all(_device_run("layernorm", x, np.array([2.0], np.float32), b).cpu().numpy() == 0.25)
    got = _device_run("rmsnorm", np.full((2, 64), 2.0, np.float32), None, None).cpu().numpy()
    assert np.allclose(got, 2.0 / np.sqrt(4.0 + 1e-5), rtol=1e-6)
    dx = torch.zeros(4, 8, device="cuda")
    assert sat.rowop_softmax(dx, 8, dx, 8, 0, 8, stream()) == 0           # no rows: nothing to do
    assert sat.rowop_softmax(dx, 4, dx, 8, 4, 8, stream()) == -1          # stride below width
    assert sat.rowop_softmax(None, 8, dx, 8, 4, 8, stream()) == -1
    assert sat.rowop_rmsnorm(dx, 40000, None, dx, 40000, 1, 32769, 1e-5, stream()) == -1   # too wide


@pytest.mark.parametrize("i", range(60))
def test_random_rows_strides_and_offsets(i):
    # Seeded random rows x width, row strides (ldx, ldy >= width) and float
    # offsets of X and Y (16-byte loads only where everything allows them),
    # gamma and beta present or not; every output against the oracle, and the
    # padding around Y untouched.
    rng = np.random.default_rng(7000 + i)
    op = si.ROWOPS[i % 3]
    rows = int(rng.integers(1, 300))
    width = int(rng.integers(1, 20000)) if i % 4 else int(rng.integers(1, 600))
    ldx, ldy = width + int(rng.integers(0, 9)), width + int(rng.integers(0, 9))
    ox, oy = int(rng.integers(0, 4)), int(rng.integers(0, 4))
    x, g, b = si.rowop_inputs(rows, width, seed=40 + i)
    if rng.integers(0, 2):
        g = None
    if rng.integers(0, 2):
        b = None
    fx = np.zeros(ox + rows * ldx + 4, np.float32)
    fx[ox:ox + rows * ldx].reshape(rows, ldx)[:, :width] = x
    fy = np.full(oy + rows * ldy + 4, -777.0, np.float32)
    dx, dy = torch.from_numpy(fx).cuda(), torch.from_numpy(fy).cuda()
    dg = torch.from_numpy(g).cuda() if g is not None else None
    db = torch.from_numpy(b).cuda() if b is not None else None
    px, py = dx.data_ptr() + 4 * ox, dy.data_ptr() + 4 * oy
    if op == "softmax":
        rc = sat.rowop_softmax(px, ldx, py, ldy, rows, width, stream())
    elif op == "rmsnorm":
        rc = sat.rowop_rmsnorm(px, ldx, dg, py, ldy, rows, width, 1e-5, stream())
    else:
        rc = sat.rowop_layernorm(px, ldx, dg, db, py, ldy, rows, width, 1e-5, stream())
    assert rc == 0, sat.gemm_last_error()
    torch.cuda.synchronize()
    out = dy.cpu().numpy()
    view = out[oy:oy + rows * ldy].reshape(rows, ldy)
    what = f"{op} rows={rows} width={width} ldx={ldx} ldy={ldy} offsets={ox},{oy} gamma={g is not None} beta={b is not None}"
    assert np.all(out[:oy] == -777.0) and np.all(out[oy + rows * ldy:] == -777.0), f"outside Y: {what}"
    assert np.all(view[:, width:] == -777.0), f"Y padding written: {what}"
    ref = oracle.softmax(x) if op == "softmax" else oracle.rmsnorm(x, g) if op == "rmsnorm" else \
        oracle.layernorm(x, g, b)
    _check(op, view[:, :width], ref, what)
