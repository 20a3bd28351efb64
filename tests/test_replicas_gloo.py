"""Replica timing across ranks (CPU, gloo, world size 2).

The path does not shard (layers are sequential and a layer's K/V is a few MB),
so N GPUs run N independent replicas; the only cross-rank steps are a barrier
and the MAX of the per-rank times.  This runs that reduction on two CPU
processes.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [12.5, 20.0][rank]
        ms = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
        q.put((rank, ms, bench.replica_throughput(100, world, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, value in got:
        assert ms == 20.0                       # the slower rank sets the time
        assert value == pytest.approx(100 * 2 / 0.020)   # units of both ranks


def test_single_rank_is_unchanged():
    import bench
    assert bench.max_over_ranks(7.5, 1, None) == 7.5
    assert bench.replica_throughput(30, 1, 10.0) == pytest.approx(3000.0)
