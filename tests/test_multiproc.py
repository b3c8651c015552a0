"""The N-replica path of bench.py on CPU: world size 2 over gloo (127.0.0.1).
Replicas exchange nothing but the slowest rank's time; the reference arm runs
on rank 0 only."""
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


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.job_time_ms(10.0 + 5.0 * rank, dist, "cpu")
    out[rank] = ms
    dist.destroy_process_group()


def test_job_time_is_the_slowest_rank():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_process_time_is_local():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.job_time_ms(3.5) == 3.5


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun every rank but 0 exits 0 without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
