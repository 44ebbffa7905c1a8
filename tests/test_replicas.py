"""bench.py with more than one process, on the CPU.

The decode has no exchange step, so a multi-GPU run is N independent replicas:
each rank times its own steps, the job's time is the slowest rank's, and the
job's throughput counts the bytes of every replica.  These tests run that host
logic as two gloo ranks, and check that the reference arm prints from rank 0
only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took 1 + r ms per step and 10 + 5 r ms end to end
        ms = bench.max_over_ranks(1.0 + rank, dist, "cpu")
        e2e = bench.max_over_ranks(10.0 + 5 * rank, dist, "cpu")
        results[rank] = (ms, e2e, bench.whole_job_gbs(1e9, world, ms))
    finally:
        dist.destroy_process_group()


def test_replica_timing_is_the_slowest_rank_and_value_counts_every_replica():
    import torch.multiprocessing as mp
    world = 2
    with mp.get_context("spawn").Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        got = dict(results)
    assert sorted(got) == [0, 1]
    for r in range(world):
        ms, e2e, gbs = got[r]
        assert ms == 2.0 and e2e == 15.0
        # 1 GB per replica, two replicas, 2 ms per step
        assert gbs == pytest.approx(1000.0)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.whole_job_gbs(2e9, 1, 4.0) == pytest.approx(500.0)


def _reference_arm(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config",
         "tiny", "--steps", "3", "--warmup", "1", "--gpus", str(world)],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_on_rank_zero_only():
    other = _reference_arm(1, 2)
    assert other.returncode == 0, other.stderr
    assert other.stdout.strip() == ""
    first = _reference_arm(0, 2)
    assert first.returncode == 0, first.stderr
    lines = [ln for ln in first.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["steps"] == 3
    assert rec["value"] > 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
