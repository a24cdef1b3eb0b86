"""The multi-rank path of bench.py on CPU: two gloo ranks take the slowest rank's time and
report the whole job's rate; the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) * 10 ms for its steps: the job's time is the slowest rank's
        total = bench.max_over_ranks(10.0 * (rank + 1), world, torch.device("cpu"))
        rate = bench.job_rate(world, 512, 4, total)
        assert bench.dist_env() == (rank, world, rank)
        out.put((rank, total, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_and_sum_the_batches():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(out.get(timeout=10) for _ in range(2))
    for rank, total, rate in res:
        assert total == 20.0
        assert rate == pytest.approx(2 * 512 * 4 / 0.020)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.job_rate(1, 64, 10, 100.0) == pytest.approx(6400.0)


def test_reference_arm_runs_on_rank_zero_only():
    import subprocess

    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "layer",
                        "--gpus", "2", "--steps", "1", "--warmup", "1"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
