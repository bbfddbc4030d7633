"""Replica aggregation of the benchmark across ranks (CPU, gloo, world size 2).

The cache does not shard: N GPUs run N independent replicas, and the whole-job number
is the bytes of all ranks over the slowest rank's time. This checks that reduction
(sum of bytes, max of seconds) with two real gloo ranks on 127.0.0.1.
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


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    b, s = bench.aggregate(dist, 100.0 * (rank + 1), 0.5 + rank, device="cpu")
    out[rank] = (b, s)
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    os.environ["PYTHONPATH"] = root + os.pathsep + os.environ.get("PYTHONPATH", "")
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == (300.0, 1.5)


def test_aggregate_single_process_is_identity():
    import bench

    assert bench.aggregate(None, 12.0, 3.0) == (12.0, 3.0)
