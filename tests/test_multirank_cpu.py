"""The benchmark's multi-rank host logic on CPU: two gloo ranks, no GPU.

Each rank runs its own batch (weak scaling, no collective on the data path);
only the timing is reduced (max over ranks) and the job bandwidth counts the
bytes of every rank over the slowest rank's step time.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from paged_kv_cache_62_gb300 import workloads
        seed = bench.rank_seed("tiny", rank)
        wl = workloads.make("tiny", "cpu", seed=seed)
        ms = 1.0 + rank                       # rank 1 is the slow one
        slow = bench.reduce_over_ranks(ms, "max", "cpu")
        fast = bench.reduce_over_ranks(ms, "min", "cpu")
        q_sum = float(wl.layers[0].q.float().sum())
        out[rank] = (seed, slow, fast, q_sum, bench.job_bandwidth(1_000_000, world, slow))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    (s0, slow0, fast0, q0, bw0), (s1, slow1, fast1, q1, bw1) = res[0], res[1]
    assert s0 != s1 and q0 != q1            # different batches per rank
    assert slow0 == slow1 == 2.0 and fast0 == fast1 == 1.0
    assert bw0 == pytest.approx(2 * 1_000_000 / 2e-3 / 1e9)


def test_single_process_reduce_is_identity():
    import bench
    assert bench.reduce_over_ranks(3.5, "max", "cpu") == 3.5
