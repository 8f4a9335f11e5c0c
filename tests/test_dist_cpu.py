"""The multi-rank plumbing of bench.py on CPU: two gloo ranks, each with its
own shard of requests (weak scaling), meet only at the barrier and the
max/sum of their timings; no collective touches the data path."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    d = bench.Dist()
    try:
        d.barrier()
        mx = d.max(float(rank + 1) * 10.0)
        sm = d.sum(64.0)
        seed = bench.shard_seed(1002, rank)
        out.put((rank, mx, sm, seed))
    finally:
        d.close()


def test_two_gloo_ranks_shard_and_reduce_timings():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r[1] for r in res] == [20.0, 20.0]      # max over ranks
    assert [r[2] for r in res] == [128.0, 128.0]    # total tokens over ranks
    assert res[0][3] != res[1][3]                   # each rank draws its own requests
