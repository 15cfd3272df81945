"""World-size-2 CPU (gloo) check of the bench's multi-rank host logic: each
rank owns a disjoint batch of sequences (weak scaling, no data-path
collective) and the step time reported is the max over ranks."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    seqs = bench.rank_sequences(r, 32)
    got = bench.reduce_max(1.5 + r, w)           # rank 1 is slower
    gathered = [None] * world
    dist.all_gather_object(gathered, seqs)
    q.put((r, w, lr, got, gathered))
    dist.destroy_process_group()


def test_two_ranks_shard_sequences_and_take_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, lr, got, gathered in res:
        assert w == 2 and lr == r
        assert got == 2.5
        a, b = gathered
        assert len(a) == len(b) == 32 and not set(a) & set(b)
        assert sorted(a + b) == list(range(64))
