"""bench.py's launch rules, checked on the host without a GPU.

The multiply has no exchange step, so the benchmark is a single-GPU program:
asked for more than one GPU, or started as one rank of several, it refuses
with a message instead of quietly measuring one GPU. The reference arm (the
CPU oracle) runs on rank 0 alone; its other ranks exit 0 without output.
"""
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BENCH = os.path.join(ROOT, "bench.py")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_more_than_one_gpu_is_refused():
    r = subprocess.run([sys.executable, BENCH, "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 2
    assert r.stdout.strip() == ""
    assert "single-GPU design" in r.stderr


def test_two_ranks_under_torchrun_are_refused():
    # The launch the contract uses for N > 1, with two CPU processes: every
    # rank refuses, so torchrun reports failure and nothing is printed.
    port = _free_port()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                        str(port), BENCH, "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode != 0
    assert '"metric"' not in r.stdout
    assert "single-GPU design" in r.stderr


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, BENCH, "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
