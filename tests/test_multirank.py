"""The whole-job throughput of a multi-GPU bench run, on CPU ranks (gloo,
world size 2): every rank times its own replica of the workload, the job time
is the slowest rank's, and the job's frames are all ranks' frames."""

import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import sys

    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.job_throughput(times[rank], 10, 1000, world, "cpu")
    finally:
        dist.destroy_process_group()


def test_job_throughput_takes_the_slowest_rank_and_all_frames():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, [12.0, 20.0], out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(2):
            ms, value = out[r]
            assert ms == pytest.approx(2.0)  # 20 ms over 10 steps, the slower rank
            assert value == pytest.approx(2 * 1000 / 2e-3)


def test_single_rank_needs_no_process_group():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    ms, value = bench.job_throughput(30.0, 10, 500, 1)
    assert ms == pytest.approx(3.0)
    assert value == pytest.approx(500 / 3e-3)
