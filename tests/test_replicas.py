"""The multi-GPU path, on the CPU with gloo ranks (world size 2).

The decode path shards by request: each replica holds its own requests' KV,
sketches and tiers and runs the whole step alone, with no exchange.  The one
collective is the bench's: the job's time is the slowest replica's (a max over
the ranks, outside the timed region), and the job's throughput is the units
all replicas processed over that time.  These tests run that host logic as
two gloo processes, and check that the reference arm works on rank 0 only.
"""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, world)            # rank 1 is the slow replica
        e2e = bench.max_over_ranks([0.5, 0.25][rank], world)
        rate = bench.job_rate(200 * 16, ms * 1e-3, world)
        with open(os.path.join(out_dir, f"{rank}.txt"), "w") as f:
            f.write(f"{ms!r} {e2e!r} {rate!r}")
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_time(tmp_path):
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        ms, e2e, rate = map(float, (tmp_path / f"{r}.txt").read_text().split())
        assert ms == 15.0 and e2e == 0.5                 # every rank sees the max
        assert rate == pytest.approx(2 * 200 * 16 / 0.015)


def test_single_replica_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_rate(16, 0.002, 1) == pytest.approx(8000.0)


def test_reference_arm_prints_on_rank_0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""
