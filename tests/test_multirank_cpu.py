"""World-size-2 CPU (gloo) checks of the multi-rank host logic:

* the bench's sequence sharding: each rank owns a disjoint batch of
  sequences (weak scaling, no data-path collective) and the step time
  reported is the max over ranks;
* the context-sharded decode step: each rank owns half of every sequence's
  entries, exchanges Top-K candidates and partial attention outputs by
  all-gather, and every rank ends with the unsharded step's result (the
  phase steps run on the CPU oracle)."""

import os
import socket
import sys

import numpy as np

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


def _shard_worker(rank, world, port, pool, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from fp4_kv_cache_02_gb300.sharding import ShardPlan, TorchComm, decode_step
    from helpers import DecodeCase
    from oracle_ops import OracleOps, shard_inputs
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        if pool:
            case = DecodeCase(workload=98, Ns=[2048, 1100], n_swa=8, reindex=True, planted_blocks=6)
        else:
            case = DecodeCase(workload=97, Ns=[2048, 1500, 300], L=2, n_swa=16)
        plan = ShardPlan(case.cap, world)
        x = shard_inputs(case, plan, rank, reindex=pool)
        res = decode_step(OracleOps(), TorchComm(), plan, rank, x, k=64 if pool else 128,
                          pool_blocks=32 if pool else 0)
        q.put((rank, [t.numpy() for t in res]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("pool,world", [(False, 2), (True, 2), (False, 3), (True, 3)])
def test_ranks_context_sharded_step_equals_unsharded(pool, world):
    """2 or 3 gloo ranks; with 3 the 128-aligned ranges are uneven and a short
    sequence has no visible entry on the later ranks."""
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from helpers import DecodeCase
    from oracle_ops import unsharded_reference
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, world, port, pool, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    if pool:
        case = DecodeCase(workload=98, Ns=[2048, 1100], n_swa=8, reindex=True, planted_blocks=6)
        ref_idx, ref_out, ref_full = unsharded_reference(case, 64, pool_blocks=32)
    else:
        case = DecodeCase(workload=97, Ns=[2048, 1500, 300], L=2, n_swa=16)
        ref_idx, ref_out, ref_full = unsharded_reference(case, 128)
    for r in range(world):
        idx, out = res[r][0], res[r][1]
        assert np.array_equal(idx, ref_idx)
        np.testing.assert_allclose(out, ref_out, rtol=1e-11, atol=1e-12)
        if pool:
            assert np.array_equal(res[r][4], ref_full)
        assert np.array_equal(res[0][1], res[r][1])  # every rank holds the same merged output
