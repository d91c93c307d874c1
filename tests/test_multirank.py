"""Host logic of the multi-rank benchmark on CPU: world_size 2 over gloo.
Each rank owns a disjoint shard of sequences (weak scaling, no data-path
collective); the timed interval is reduced with max over ranks."""
import os
import socket

import pytest
import torch
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, wsz, local = bench.dist_env()
        shard = list(bench.shard_sequences(8, wsz, r))
        t = bench.max_over_ranks(1.5 + r, wsz)  # rank 1 is the slow one
        bench.barrier(wsz)
        gathered = [None] * wsz
        dist.all_gather_object(gathered, shard)
        q.put((r, shard, t, gathered, bench.rank_seed(100, r)))
    finally:
        dist.destroy_process_group()


def test_two_rank_sharding_and_timing():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    shards = [r[1] for r in res]
    assert shards[0] == list(range(0, 8)) and shards[1] == list(range(8, 16))
    assert not set(shards[0]) & set(shards[1])
    assert all(r[2] == 2.5 for r in res)          # max over ranks
    assert res[0][3] == res[1][3] == shards       # every rank sees the same partition
    assert res[0][4] != res[1][4]                 # distinct data per rank
