"""The N > 1 host logic of bench.py on CPU with the gloo backend, world size 2: the job
time is the slowest rank's, the job rate counts every rank's units, each rank draws its
own batch, and only rank 0 runs the reference arm."""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    from selective_scan_mamba_gb300 import synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = 0.001 * (rank + 1)  # rank 1 is the slower one
        t_max = bench.max_over_ranks(dist, t, "cpu")
        rate = bench.whole_job_rate(100, world, t_max)
        x = synth.mamba1(1, 4, 16, 8, seed=rank).arrays["x"]  # the seed the bench uses per rank
        gathered = [None] * world
        dist.all_gather_object(gathered, x.tolist())
        out.put((rank, t_max, rate, gathered))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t_max, rate, gathered in res:
        assert t_max == pytest.approx(0.002)          # the slowest rank's time, on every rank
        assert rate == pytest.approx(100 * 2 / 0.002)  # all ranks' units over that time
        assert not np.array_equal(np.array(gathered[0]), np.array(gathered[1]))  # own batches


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import argparse

    import bench
    args = argparse.Namespace(steps=1, warmup=0, cpu_seconds=0.1)
    assert bench.bench_reference(args, 1, 2) is None


def test_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 0.5, "cpu") == 0.5
    assert bench.whole_job_rate(10, 1, 2.0) == 5.0
