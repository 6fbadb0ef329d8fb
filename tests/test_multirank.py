"""The N > 1 path of the benchmark without a GPU: two gloo ranks on the host.

One process per GPU runs an independent replica (the multiply has no exchange
step), the job's time is the slowest replica's, and the whole-job value is the
work of all replicas over that time. The reference arm runs on rank 0 alone.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        local = [3.0, 5.0][rank]  # the second replica is slower
        t = bench.max_over_ranks(local, world, "cpu")
        out[rank] = (t, bench.job_tflops(world, 2e12, 10, t))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time_and_all_work_counts():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1]
    t, v = out[0]
    assert t == 5.0
    assert v == pytest.approx(world * 2e12 * 10 / 5e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.0, 1) == 4.0
    assert bench.job_tflops(1, 1e12, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
