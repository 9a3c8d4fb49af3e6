"""On-device sweep of every candidate (tile, schedule) for GEMM shapes.

For each shape and dtype, every configuration the kernels support (tile N,
single SM or CTA pair, raster order, raster group) is timed the way the
benchmark times the dispatcher's choice: L2 flushed by a 256 MiB write
before each run, a CUDA event pair around each gemm_run, median of the
timed runs. Results go to a JSON file; ``--table`` also writes the winners
as the dispatcher's committed table (``csrc/sweep_table.inc``).

This is the offline counterpart of the tactic ranking in the FlashInfer
pull request "fix(fp4_gemm autotune) SM107 kernel family excluded from
autotune candidates": measure every candidate instead of truncating a
scored list, then freeze the winners so that the runtime does no tuning.

  python -m shape_adaptive_tile_gb300.sweep --out sweep.json [--table] [--shapes tf32:2048x2048x2048 ...]
"""
from __future__ import annotations

import argparse
import itertools
import json
import os
import re
import statistics
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
TABLE = os.path.join(HERE, "csrc", "sweep_table.inc")
DT_CODE = {"tf32": 0, "bf16": 1, "fp16": 2}


def candidates(M, N, K, dtype, tma_ok, sm_count=152, beta=0.0):
    out = []
    kb = -(-K // (32 if dtype == "tf32" else 64))
    for bn, cg in ((256, 2), (128, 2), (256, 1), (128, 1), (64, 1)):
        # Rows TMA cannot address directly take the class-view tiles (1-SM
        # 128 or 256 columns, CTA-pair 256), compared with the plain loads.
        if not tma_ok and (bn == 64 or (cg == 2 and bn != 256)):
            continue
        if cg == 2 and M <= 128:
            continue
        tiles = -(-M // (128 * cg)) * -(-N // bn)
        slots = sm_count // cg
        for raster, group in itertools.product((0, 1), (1, 2, 4, 8, 16)):
            out.append(f"{bn},{cg},{raster},{group}")
            # stream-K where more than a wave of tiles ends in a partial one
            if tiles > slots and tiles % slots:
                out.append(f"{bn},{cg},{raster},{group},sk")
            # beta != 0: also with the epilogue loading C itself instead of
            # the producer fetching it through the ring (the 1-SM 256-wide
            # tile has no ring stages to spare, so it always loads C itself)
            if beta != 0.0 and tma_ok and (bn, cg) != (256, 1):
                out.append(f"{bn},{cg},{raster},{group},cload")
        if not tma_ok and cg == 1:
            for raster, group in itertools.product((0, 1), (2, 4)):
                out.append(f"{bn},{cg},{raster},{group},plain")
        # K splits only where the tiles alone leave at least half the SMs idle
        ctas = -(-M // (128 * cg)) * -(-N // bn) * cg
        for s in (2, 4, 8):
            if ctas * s <= 2 * sm_count and kb // s >= 4:
                for group in (2, 8):
                    out.append(f"{bn},{cg},0,{group},{s}")
    # Skinny M: operand roles exchanged, tiles of 128 columns by bn rows of C.
    if tma_ok and M <= 128:
        for bn in (32, 64, 128):
            if bn > 2 * M and bn > 32:
                continue
            tiles = -(-N // 128) * -(-M // bn)
            for raster, group in itertools.product((0, 1), (2, 8)):
                out.append(f"{bn},1,{raster},{group},swap")
            for s in (2, 4, 8):
                if tiles * s <= 2 * sm_count and kb // s >= 4:
                    out.append(f"{bn},1,0,8,{s},swap")
    return out


# Shallower ring depths compiled for the untransposed TMA tiles, by (bn, cg).
ALT_STAGES = {(64, 1): 4, (128, 1): 4, (256, 1): 3, (128, 2): 4, (256, 2): 4}


def stage_variants(config):
    """The configuration with each other compiled ring depth (",st<n>"), for
    untransposed TMA tiles; none for plain-load or swapped ones."""
    parts = config.split(",")
    if "plain" in parts or "swap" in parts:
        return []
    alt = ALT_STAGES.get((int(parts[0]), int(parts[1])))
    return [f"{config},st{alt}"] if alt else []


def time_config(sat, torch, M, N, K, dtype, config, dA, dB, dC, flush, runs, warmup, alpha=1.0, beta=0.0):
    stream = torch.cuda.current_stream()
    with sat.Plan(M, N, K, dtype, config) as plan:
        for _ in range(warmup):
            plan.run(dA, dB, dC, alpha, beta, stream.cuda_stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(runs)]
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            plan.run(dA, dB, dC, alpha, beta, stream.cuda_stream)
            e1.record(stream)
        torch.cuda.synchronize()
        sat.check(plan.status())
        t = sorted(e0.elapsed_time(e1) for e0, e1 in ev)
        return {"config": config, "plan": plan.describe(), "median_ms": statistics.median(t), "min_ms": t[0]}


def sweep_shape(sat, torch, M, N, K, dtype, runs=30, warmup=3, configs=None, alpha=1.0, beta=0.0):
    es = 4 if dtype == "tf32" else 2
    tma_ok = (K * es) % 16 == 0 and (N * es) % 16 == 0
    rng = np.random.default_rng(0)
    tdt = {"tf32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    dA = torch.from_numpy(rng.integers(-4, 5, (M, K)).astype(np.float32)).to("cuda", tdt)
    dB = torch.from_numpy(rng.integers(-4, 5, (K, N)).astype(np.float32)).to("cuda", tdt)
    # C starts finite; with beta != 0 it is read (and C = alpha*A*B + beta*C stays bounded).
    dC = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32)).to("cuda")
    flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
    res = []

    def run(cfg):
        r = time_config(sat, torch, M, N, K, dtype, cfg, dA, dB, dC, flush, runs, warmup, alpha, beta)
        r["tflops"] = 2.0 * M * N * K / (r["median_ms"] * 1e-3) / 1e12
        res.append(r)

    for cfg in configs or candidates(M, N, K, dtype, tma_ok, beta=beta):
        run(cfg)
    # Ring depth, the last dimension: the three fastest configurations again
    # with each shallower compiled ring.
    if tma_ok and not configs:
        for best in sorted(res, key=lambda r: r["median_ms"])[:3]:
            for cfg in stage_variants(best["config"]):
                run(cfg)
    with sat.Plan(M, N, K, dtype) as p:
        chosen = p.describe()
    return {"dtype": dtype, "M": M, "N": N, "K": K, "alpha": alpha, "beta": beta, "results": res,
            "dispatcher": chosen}


def table_row(e):
    """The table line for one swept shape: its fastest configuration."""
    best = min(e["results"], key=lambda r: r["median_ms"])
    parts = best["config"].split(",")
    bn, cg, raster, group = parts[:4]
    nums = [p for p in parts[4:] if p.isdigit()]
    splits = nums[0] if nums else "1"
    cload = 1 if "cload" in parts[4:] else 0
    sk = 1 if "sk" in parts[4:] else 0
    swap = 1 if "swap" in parts[4:] else 0
    stages = next((int(p[2:]) for p in parts[4:] if p.startswith("st") and p[2:].isdigit()), 0)
    return (f"{{{DT_CODE[e['dtype']]}, {e['M']}, {e['N']}, {e['K']}, {{{bn}, {cg}, {raster}, {group}, 0, {splits}, "
            f"{cload}, {sk}, {swap}, {stages}}}}},  // {best['tflops']:.1f} TFLOP/s, {best['median_ms'] * 1e3:.1f} us")


def _key(line):
    m = re.match(r"\{(-?\d+), (\d+), (\d+), (\d+),", line)
    return tuple(int(x) for x in m.groups()) if m else None


def write_table(entries, path=TABLE, merge=False):
    """Write the winners as the dispatcher's table; with `merge`, rows of the
    existing table for shapes not swept now are kept."""
    rows = {}
    if merge and os.path.exists(path):
        with open(path) as f:
            for line in f:
                k = _key(line)
                if k and k[0] >= 0:
                    rows[k] = line.rstrip("\n")
    for e in entries:
        rows[(DT_CODE[e["dtype"]], e["M"], e["N"], e["K"])] = table_row(e)
    lines = ["// Committed sweep table: {dtype, M, N, K, {bn, cg, raster, group, 0, splits, cload, sk, swap, stages}}.",
             "// Written by shape_adaptive_tile_gb300/sweep.py from on-device timings",
             "// (median of L2-flushed runs) of every candidate configuration."]
    order = {1: 0, 2: 1, 0: 2}  # bf16, fp16, tf32
    lines += [rows[k] for k in sorted(rows, key=lambda k: (order[k[0]], k[1:]))]
    lines.append("{-1, 0, 0, 0, {256, 1, 0, 8, 0}},")
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", required=True)
    ap.add_argument("--shapes", nargs="*",
                    help="dtype:MxNxK[:beta] (default: every benchmark workload, with its own alpha and beta)")
    ap.add_argument("--configs", nargs="*", help="restrict to these configurations")
    ap.add_argument("--runs", type=int, default=30)
    ap.add_argument("--table", action="store_true", help="also write csrc/sweep_table.inc")
    ap.add_argument("--merge", action="store_true", help="with --table: keep the rows of shapes not swept now")
    args = ap.parse_args(argv)
    sys.path.insert(0, os.path.dirname(HERE))
    import torch
    import shape_adaptive_tile_gb300 as sat
    import synth_inputs as si
    torch.cuda.set_device(0)
    sat.build()
    if args.shapes:
        shapes = []
        for s in args.shapes:
            parts = s.split(":")
            beta = float(parts[2]) if len(parts) > 2 else 0.0
            shapes.append((parts[0], tuple(int(x) for x in parts[1].split("x")), 1.0 if beta == 0 else 1.5, beta))
    else:
        shapes = sorted({(w[1], w[2], w[4], w[5]) for w in si.WORKLOADS})
    entries = []
    for dt, (M, N, K), alpha, beta in shapes:
        e = sweep_shape(sat, torch, M, N, K, dt, args.runs, configs=args.configs, alpha=alpha, beta=beta)
        best = min(e["results"], key=lambda r: r["median_ms"])
        print(f"{dt} {M}x{N}x{K} beta {beta:g}: best {best['config']} {best['tflops']:.1f} TFLOP/s; "
              f"dispatcher [{e['dispatcher']}]", flush=True)
        for r in sorted(e["results"], key=lambda r: r["median_ms"])[:5]:
            print(f"    {r['config']:>12} {r['median_ms'] * 1e3:9.1f} us {r['tflops']:8.1f} TFLOP/s", flush=True)
        entries.append(e)
        with open(args.out, "w") as f:
            json.dump(entries, f, indent=1)
    if args.table:
        write_table(entries, merge=args.merge)


if __name__ == "__main__":
    main()
