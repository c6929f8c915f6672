"""The N > 1 path of bench.py on CPU: two gloo ranks.  Every rank streams its
own replica (no collective on the data path); the job's time is the slowest
rank's and the whole-job throughput counts every rank's bytes."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench._dist() == (world, rank, rank)
        local_ms = [40.0, 55.5][rank]  # the second replica is the slower one
        ms = bench._max_over_ranks(local_ms, world, torch.device("cpu"))
        value = bench._job_throughput(world, 536870912, ms / 100)
        dist.barrier()
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in res:
        assert ms == 55.5  # max over ranks, identical on both
        assert value == pytest.approx(2 * 536870912 / (0.555e-3) / 1e9)


def test_single_rank_needs_no_collective():
    import bench

    assert bench._max_over_ranks(12.5, 1, torch.device("cpu")) == 12.5
    assert bench._job_throughput(1, 1000, 1.0) == pytest.approx(1e-3)


def test_reference_arm_under_two_ranks_prints_only_on_rank_0():
    # rank 1 of a torchrun launch must exit 0 without work or output
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
