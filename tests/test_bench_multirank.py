"""The benchmark's multi-rank host logic on CPU: two gloo ranks, no GPU.

Each rank runs its own replica; the job time is the slowest rank's and the
reported throughput counts every rank's bytes.  The reference arm prints from
rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [0.25, 0.40][rank]                     # rank 1 is the slower one
    job_ms = bench.max_over_ranks(local_ms, world)
    gbs = bench.job_throughput(1_000_000_000, world, job_ms)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"job_ms": job_ms, "gbs": gbs}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r in res:
        assert r["job_ms"] == pytest.approx(0.40)
        assert r["gbs"] == pytest.approx(2 * 1.0 / 0.40e-3)   # 2 ranks x 1 GB per 0.4 ms


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.job_throughput(2e9, 1, 1.0) == pytest.approx(2000.0)


def test_reference_arm_prints_from_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, env=env,
                         timeout=600)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_reference_arm_stays_within_its_budget():
    """The reference arm (the fp64 oracle on the host cores) cuts each group to a sequence
    prefix when the requested steps would take longer than its budget, and says so."""
    import argparse
    import time
    sys.path.insert(0, ROOT)
    import bench
    args = argparse.Namespace(steps=40, warmup=3)
    t0 = time.perf_counter()
    line = bench.run_reference(args, budget_s=4.0)
    oracle_s = time.perf_counter() - t0
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 40
    assert line["config"]["workload"] == bench.LONG_WORKLOAD
    assert "the first" in line["cpu_baseline"]["sample"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert oracle_s < 120  # data generation plus about the budget
