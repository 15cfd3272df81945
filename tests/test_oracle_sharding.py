"""Pins of the oracle's merge steps for a context-sharded decode step, and
the sharding host logic run on CPU ranks in turn.

The attention merge is pinned to the oracle's attention on the union of the
row sets (a different function), Top-K merging to the unsharded Top-K, the
block maxima to a numpy brute force."""

import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_02_gb300.inputs import bf16_round
from fp4_kv_cache_02_gb300.sharding import ShardPlan, sequential_decode_step

from helpers import DecodeCase
from oracle_ops import OracleOps, shard_inputs, unsharded_reference


def _kv(rng, n):
    return oracle.pack_kv_fp4(bf16_round(rng.standard_normal((n, 512)).astype(np.float32)))


@pytest.mark.parametrize("cuts", [[0, 40], [0, 17, 40], [0, 0, 25, 40], [0, 1, 2, 40]])
def test_attn_merge_of_disjoint_sets_is_attention_on_the_union(cuts):
    rng = np.random.default_rng(7)
    kd, ks = _kv(rng, 60)
    swa = oracle.pack_fp8(bf16_round(rng.standard_normal((6, 512)).astype(np.float32)))
    q = bf16_round(rng.standard_normal((5, 512)).astype(np.float32) * 0.08)
    idx = rng.permutation(60)[:40].astype(np.int32)
    full, full_lse = oracle.sparse_attn(q, kd, ks, idx, swa)
    outs, lses = [], []
    for r in range(len(cuts) - 1):
        part = np.full(40, -1, np.int32)
        part[cuts[r]:cuts[r + 1]] = idx[cuts[r]:cuts[r + 1]]
        o, l = oracle.sparse_attn(q, kd, ks, part, swa if r == len(cuts) - 2 else None)
        outs.append(o)
        lses.append(l)
    out, lse = oracle.attn_merge(np.stack(outs), np.stack(lses))
    np.testing.assert_allclose(out, full, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, full_lse, rtol=1e-13)
    # rank order does not change the merged value
    out2, lse2 = oracle.attn_merge(np.stack(outs[::-1]), np.stack(lses[::-1]))
    np.testing.assert_allclose(out2, full, rtol=1e-12, atol=1e-13)


def test_attn_merge_special_cases():
    rng = np.random.default_rng(8)
    o = rng.standard_normal((1, 3, 4))
    l = rng.standard_normal((1, 3))
    out, lse = oracle.attn_merge(o, l)                      # one set: itself
    assert np.array_equal(out, o[0]) and np.array_equal(lse, l[0])
    ninf = np.full((1, 3), -np.inf)
    out, lse = oracle.attn_merge(np.concatenate([o, 5 * o]), np.concatenate([l, ninf]))
    np.testing.assert_allclose(out, o[0], rtol=1e-15)       # an empty set adds nothing
    np.testing.assert_allclose(lse, l[0], rtol=1e-15)
    out, lse = oracle.attn_merge(np.zeros((2, 3, 4)), np.full((2, 3), -np.inf))
    assert np.all(out == 0) and np.all(lse == -np.inf)     # no rows anywhere
    # two equal-mass sets: the mean of the outputs, lse + log 2
    out, lse = oracle.attn_merge(np.stack([o[0], -o[0] + 1]), np.stack([l[0], l[0]]))
    np.testing.assert_allclose(out, np.full((3, 4), 0.5), rtol=1e-15)
    np.testing.assert_allclose(lse, l[0] + np.log(2), rtol=1e-15)


@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 64, 1001])
def test_block_max_brute_force(n):
    rng = np.random.default_rng(n)
    s = rng.standard_normal(n).astype(np.float32)
    if n > 3:
        s[1] = np.nan
        s[2] = -np.inf
    got = oracle.block_max(s, 8)
    assert got.shape == (-(-n // 8),)
    for j in range(got.size):
        blk = s[8 * j:8 * j + 8]
        blk = blk[~np.isnan(blk)]
        assert got[j] == (blk.max() if blk.size else -np.inf)


def test_shard_plan_covers_the_capacity_with_aligned_disjoint_ranges():
    for cap in (0, 128, 1000, 65536, 65536 + 128):
        for world in (1, 2, 3, 4, 8):
            plan = ShardPlan(cap, world)
            b = plan.all_bounds()
            assert b[0][0] == 0 and b[-1][1] == cap
            for (lo, hi), (lo2, _) in zip(b, b[1:]):
                assert hi == lo2 and lo % 128 == 0 and lo <= hi
            nv = [0, cap // 3, cap]
            assert [sum(x) for x in zip(*[plan.local_visible(r, nv) for r in range(world)])] == nv
    with pytest.raises(ValueError):
        ShardPlan(100, 2, align=12)


def test_topk_merge_of_shard_candidates_is_the_global_topk():
    rng = np.random.default_rng(9)
    n, k = 5000, 300
    s = rng.standard_normal(n).astype(np.float32)
    s[100:140] = 2.5                                     # ties across a shard bound
    ref, _ = oracle.topk(s, k)
    vals, pos = [], []
    for lo, hi in ShardPlan(n, 3).all_bounds():
        loc, _ = oracle.topk(s[lo:hi], k)
        vals.append(np.where(loc >= 0, s[lo:hi][np.maximum(loc, 0)], -np.inf).astype(np.float32))
        pos.append(np.where(loc >= 0, loc + lo, -1).astype(np.int32))
    got, _ = oracle.topk(np.concatenate(vals), k, positions=np.concatenate(pos))
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("world", [1, 2, 3])
def test_sequential_sharded_step_equals_the_unsharded_oracle(world):
    case = DecodeCase(workload=97, Ns=[2048, 1500, 300], L=2, n_swa=16)
    plan = ShardPlan(case.cap, world)
    ops = OracleOps()
    xs = [shard_inputs(case, plan, r) for r in range(world)]
    idx, out, _, lse = sequential_decode_step(ops, plan, xs, k=128)
    ref_idx, ref_out, _ = unsharded_reference(case, 128)
    assert np.array_equal(idx.numpy(), ref_idx)
    np.testing.assert_allclose(out.numpy(), ref_out, rtol=1e-11, atol=1e-12)


def test_sequential_sharded_step_with_pool_equals_the_unsharded_oracle():
    case = DecodeCase(workload=98, Ns=[2048, 1100], n_swa=8, reindex=True, planted_blocks=6)
    plan = ShardPlan(case.cap, 3)
    ops = OracleOps()
    xs = [shard_inputs(case, plan, r, reindex=True) for r in range(3)]
    idx, out, _, _, idx_full = sequential_decode_step(ops, plan, xs, k=64, pool_blocks=32)
    ref_idx, ref_out, ref_full = unsharded_reference(case, 64, pool_blocks=32)
    assert np.array_equal(idx_full.numpy(), ref_full)
    assert np.array_equal(idx.numpy(), ref_idx)
    np.testing.assert_allclose(out.numpy(), ref_out, rtol=1e-11, atol=1e-12)
