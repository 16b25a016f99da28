"""The multi-rank paths on CPU (gloo, two ranks).

Sharding: a batch is cut across ranks by sequence (K/V bytes balanced) or by
KV head, each rank decodes its share on its own -- here with the float64
oracle standing in for the GPU, which the CPU suite does not have -- the
shares are gathered and put back in batch order, and the result equals the
unsharded decode exactly.  Timing: every rank sees the slowest rank's time and
the job value counts every rank's bytes."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

F_Q4, F_Q8 = 2, 8


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run(target, world, *args):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port, q) + args) for r in range(world)]
    for pr in procs:
        pr.start()
    res = sorted((q.get(timeout=300) for _ in procs), key=lambda x: x[0])
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    return res


def _timing_worker(rank, world, port, q):
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        my_ms = 0.05 * (rank + 1)
        slowest = bench.rank_max(dist, my_ms, "cpu")
        q.put((rank, slowest, bench.job_gbps(world, 217055232, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    for rank, slowest, value in _run(_timing_worker, 2):
        assert slowest == pytest.approx(0.10)
        assert value == pytest.approx(2 * 217055232 / 0.10e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.rank_max(None, 0.07, "cpu") == 0.07
    assert bench.job_gbps(1, 217055232, 0.07) == pytest.approx(3100.79, rel=1e-4)


def _batch():
    import workloads as W
    return W.make_workload("dist", 12, [700, 33, 2000, 64, 513, 1500, 9], 16, F_Q4, F_Q8, 2, "shuffled")


def _shard_worker(rank, world, port, q, mode):
    import oracle
    import workloads as W
    from paged_kv_gqa_11_gb300 import partition as P
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        w = _batch()
        if mode == "sequence":
            parts = P.balance_by_sequence(P.kv_bytes_per_sequence(w.seq_lens, w.k_type, w.v_type), world)
            mine = w.subset(parts[rank])
        else:
            ranges = P.split_kv_heads(W.HKV, world)
            rg = ranges[rank]
            mine = W.Workload(w.name, w.seq_lens, w.n_qtok, w.page_size, w.n_blocks, w.k_type, w.v_type, w.table,
                              np.ascontiguousarray(w.k_rows[:, rg.start:rg.stop]),
                              np.ascontiguousarray(w.v_rows[:, rg.start:rg.stop]),
                              np.ascontiguousarray(w.q[:, :, P.GQA * rg.start:P.GQA * rg.stop]), w.scale)
        out, lse = oracle.decode_workload(mine)
        shares = [None] * world
        dist.all_gather_object(shares, (out, lse))
        if mode == "sequence":
            full = (P.assemble_by_sequence(parts, [s[0] for s in shares], w.n_seq),
                    P.assemble_by_sequence(parts, [s[1] for s in shares], w.n_seq))
            load = int(P.kv_bytes_per_sequence(mine.seq_lens, w.k_type, w.v_type).sum())
        else:
            full = (P.assemble_by_kv_head(ranges, [s[0] for s in shares]),
                    P.assemble_by_kv_head(ranges, [s[1] for s in shares]))
            load = mine.kv_bytes() // W.HKV * len(rg)
        q.put((rank, full, load))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("mode", ["sequence", "kv_head"])
def test_sharded_decode_equals_unsharded(mode):
    from paged_kv_gqa_11_gb300 import _build
    import oracle
    _build.build()
    oracle.build()
    res = _run(_shard_worker, 2, mode)
    want_out, want_lse = oracle.decode_workload(_batch())
    for rank, (out, lse), _ in res:
        assert np.array_equal(out, want_out) and np.array_equal(lse, want_lse), (mode, rank)
    loads = [r[2] for r in res]
    assert min(loads) > 0
    if mode == "kv_head":
        assert loads[0] == loads[1]
    else:  # longest first onto the lighter rank: within one sequence's bytes of each other
        assert abs(loads[0] - loads[1]) <= max(loads)


def test_partition_covers_every_sequence_once():
    from paged_kv_gqa_11_gb300 import partition as P
    rng = np.random.default_rng(3)
    for n_ranks in (1, 2, 3, 8):
        w = rng.integers(1, 10 ** 6, size=int(rng.integers(1, 50)))
        parts = P.balance_by_sequence(w, n_ranks)
        assert len(parts) == n_ranks
        flat = sorted(i for p in parts for i in p)
        assert flat == list(range(len(w)))
        loads = [int(w[p].sum()) for p in parts]
        # LPT bound: no rank exceeds the mean by more than the largest item
        assert max(loads) <= w.sum() / n_ranks + w.max()
    # N copies of the ragged batch: every rank gets one long and seven short
    lens = np.tile([131072] + [8192] * 7, 4)
    parts = P.balance_by_sequence(P.kv_bytes_per_sequence(lens, F_Q4, F_Q4), 4)
    for p in parts:
        assert sorted(lens[p].tolist()) == [8192] * 7 + [131072]
    with pytest.raises(ValueError):
        P.split_kv_heads(4, 3)
    with pytest.raises(ValueError):
        P.assemble_by_sequence([[0], [0]], [np.zeros((1, 2)), np.zeros((1, 2))], 2)
