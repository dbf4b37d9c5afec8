"""World-size-2 gloo tests (CPU) of the multi-GPU bench path.

The decode path shards into independent replicas (sequences are independent; no data-path
collective), so the only cross-rank steps are the timing barrier and the max over ranks of
the timed region; the whole-job throughput is the sum over replicas.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        ms = [3.0, 7.5][rank]
        got = bench.max_over_ranks(ms, torch.device("cpu"))
        dist.barrier()
        q.put((rank, got, bench._dist()[:2]))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [7.5, 7.5]
    assert [r[2] for r in res] == [(2, 0), (2, 1)]


def test_aggregate_throughput_is_weak_scaling_sum():
    import bench
    one = bench.aggregate_gbs(150_000_000, 0.04, 1)
    assert abs(one - 3750.0) < 1e-6
    assert abs(bench.aggregate_gbs(150_000_000, 0.04, 4) - 4 * one) < 1e-6
    assert bench.max_over_ranks(1.25, torch.device("cpu")) == 1.25        # no process group: identity
