"""The benchmark's multi-rank plumbing (max of elapsed time, sum of units) on CPU with gloo,
world size 2, and the JSON contract of the reference arm's sizing helpers."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier()
    t, u = bench.aggregate(10.0 + 5.0 * rank, 100.0 * (rank + 1))
    q.put((rank, t, u))
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
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
    assert res == [(0, 15.0, 300.0), (1, 15.0, 300.0)]


def test_aggregate_single_process_is_identity():
    assert bench.aggregate(3.0, 7.0) == (3.0, 7.0)
