"""The multi-rank timing path of bench.py on CPU (gloo, two ranks): every rank
sees the slowest rank's time and the job value counts every rank's bytes."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        my_ms = 0.05 * (rank + 1)
        slowest = bench.rank_max(dist, my_ms, "cpu")
        q.put((rank, slowest, bench.job_gbps(world, 217055232, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    for rank, slowest, value in res:
        assert slowest == pytest.approx(0.10)
        assert value == pytest.approx(2 * 217055232 / 0.10e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.rank_max(None, 0.07, "cpu") == 0.07
    assert bench.job_gbps(1, 217055232, 0.07) == pytest.approx(3100.79, rel=1e-4)
