"""bench.py's N > 1 path on CPU: two gloo ranks, each running its own replica.

The GEMM path has no exchange step, so N GPUs run N independent replicas
("scaling": "weak"); the job time is the slowest rank's and the job's
throughput counts the work of every rank. The reference arm under torchrun
runs on rank 0 only; other ranks exit at once without output.
"""
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, local_ms, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        job = bench.job_time_ms(local_ms[rank], world, torch)
        value, ms = bench.job_value(2.0e12, 10, job, world)
        out[rank] = (job, value, ms)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_all_work():
    world, port = 2, 29517
    local_ms = [40.0, 50.0]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, local_ms, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        job, value, ms = res[rank]
        assert job == 50.0                      # max over ranks
        assert ms == pytest.approx(5.0)         # per step
        assert value == pytest.approx(world * 2.0e12 / 5e-3 / 1e12)   # both replicas' work


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_time_ms(12.5, 1, torch) == 12.5
    value, ms = bench.job_value(1e12, 4, 8.0, 1)
    assert ms == 2.0 and value == pytest.approx(500.0)


def test_reference_arm_non_zero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_roofline_peak_follows_the_clock_record():
    # The measured bf16 figures times the nominal TF32 : BF16 ratio; the
    # sustained one only when the timed region's clock samples show the
    # power cap.
    sys.path.insert(0, ROOT)
    import bench
    pk = {"bf16_tflops": 1892.0, "bf16_tflops_sustained": 1684.0}
    capped = {"reasons": ["sw_power_cap"], "samples_in_timed_region": 12}
    peak, burst, kind = bench.roofline_peak("tf32", pk, capped)
    assert (kind, round(peak, 3), round(burst, 3)) == ("sustained", round(1684.0 * 1100 / 2250, 3),
                                                      round(1892.0 * 1100 / 2250, 3))
    for clocks in ({"reasons": [], "samples_in_timed_region": 12}, {"reasons": ["sw_power_cap"],
                                                                     "samples_in_timed_region": 0}, None):
        peak, burst, kind = bench.roofline_peak("bf16", pk, clocks)
        assert kind == "burst" and peak == burst == 1892.0
    # No sustained figure recorded: the burst one either way.
    peak, _, kind = bench.roofline_peak("fp16", {"bf16_tflops": 1900.0}, capped)
    assert kind == "burst" and peak == 1900.0
