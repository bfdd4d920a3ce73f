"""The N > 1 path of bench.py, on the CPU: replicas (one process per GPU, no
data-path collective) time with a barrier and take the slowest rank's time.

* two gloo ranks agree on the maximum of their times, and the whole-job value
  counts both ranks' bytes over that time (weak scaling);
* the reference arm under torchrun runs on rank 0 only: another rank exits 0
  and prints nothing.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        slowest = bench.max_over_ranks(times[rank], "cpu")
        out.put((rank, slowest, bench.job_value(1e9, world, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [0.002, 0.003]
    mp.start_processes(rank_main, args=(2, free_port(), times, q), nprocs=2, join=True,
                       start_method="spawn")
    got = sorted(q.get(timeout=60) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == pytest.approx(0.003)
        # both ranks' bytes (1 GB each) over the slowest time
        assert value == pytest.approx(2 * 1e9 / 0.003 / 1e9)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
