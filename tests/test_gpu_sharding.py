"""GPU parity of the context-sharding exchange steps (candidates, candidate
merge, shard positions, shard pool, block maxima, attention merge) against
their definitions and the oracle, and of a whole context-sharded decode step
run shard by shard on one GPU against the unsharded path and the oracle."""

import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_02_gb300.sharding import Csa2Ops, ShardPlan, sequential_decode_step

from helpers import ATTN_ROW_TOL, DecodeCase, attn_row_error, check_topk, dev

# sharded and unsharded steps split the same softmax into different partials;
# each rounds its P to fp16 (relative 2^-11) against its own maximum, so the
# two outputs may differ by two such roundings of the largest term
SHARD_ROW_TOL = 2 * 2.0 ** -11
from oracle_ops import shard_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    from fp4_kv_cache_02_gb300 import csa2 as m
    return m


def _sync_ok(csa2):
    torch.cuda.synchronize()
    assert csa2.csa2_get_last_error() == 0


def test_candidates_merge_and_positions_are_exact(csa2):
    rng = np.random.default_rng(21)
    R, B, n, k = 3, 4, 5000, 300
    s = rng.standard_normal((R, B, n)).astype(np.float32)
    s[0, 0, 100:140] = 3.0          # ties, straddling ranks below
    s[1, 0, 0:40] = 3.0
    s[2, 1, :] = -np.inf            # a rank with no candidates for row 1
    nvalid = np.array([n, n - 17, 0, 1], np.int32)
    pos_map = rng.permutation(n).astype(np.int32)[None, :].repeat(B, 0)
    pos_map[:, ::7] = -1
    cands, ref_vals, ref_pos = [], [], []
    for r in range(R):
        ds = dev(s[r])
        cols = torch.empty(B, k, dtype=torch.int32, device="cuda")
        csa2.csa2_topk(ds, k, cols, csa2.topk_workspace(B, n, k), n_valid=dev(nvalid))
        for use_map in (False, True):
            cand = torch.empty(B, k, 2, dtype=torch.int32, device="cuda")
            csa2.csa2_topk_candidates(ds, cols, r * n, cand, positions=dev(pos_map) if use_map else None)
            _sync_ok(csa2)
            c = cand.cpu().numpy()
            cc = cols.cpu().numpy()
            for b in range(B):
                for j in range(k):
                    col = cc[b, j]
                    p = -1 if col < 0 else (pos_map[b, col] if use_map else col)
                    if p < 0:
                        assert c[b, j, 0] == np.float32(-np.inf).view(np.int32) and c[b, j, 1] == -1
                    else:
                        assert c[b, j, 0] == s[r, b, col].view(np.int32) and c[b, j, 1] == p + r * n
            if not use_map:
                cands.append(cand)
    allc = torch.stack(cands)
    for k_out in (1, 256, 900):
        idx = torch.empty(B, k_out, dtype=torch.int32, device="cuda")
        csa2.csa2_topk_merge(allc, k_out, idx, csa2.merge_workspace(R, B, k, k_out))
        _sync_ok(csa2)
        c = allc.cpu().numpy()
        for b in range(B):
            vals = np.ascontiguousarray(c[:, b, :, 0]).view(np.float32).reshape(-1)
            pos = np.ascontiguousarray(c[:, b, :, 1]).reshape(-1)
            ref, nv = oracle.topk(vals, k_out, positions=pos)
            want = np.concatenate([np.sort(ref[:nv]), -np.ones(k_out - nv, np.int32)])
            assert np.array_equal(idx[b].cpu().numpy(), want)
    g = torch.from_numpy(rng.integers(-1, 3 * n, (B, 700)).astype(np.int32)).cuda()
    for lo, hi in ((0, n), (n, 2 * n), (2 * n - 3, 2 * n + 5), (7, 7)):
        loc = torch.empty_like(g)
        csa2.csa2_shard_positions(g, lo, hi, loc)
        _sync_ok(csa2)
        gi = g.cpu().numpy()
        assert np.array_equal(loc.cpu().numpy(), np.where((gi >= lo) & (gi < hi), gi - lo, -1))


def test_block_max_and_shard_pool_are_exact(csa2):
    rng = np.random.default_rng(22)
    B, n = 3, 4101
    s = rng.standard_normal((B, n)).astype(np.float32)
    s[0, 5] = np.nan
    s[1, 8:16] = -np.inf
    nv = np.array([n, 3000, 0], np.int32)
    bmax = torch.empty(B, -(-n // 8), dtype=torch.float32, device="cuda")
    csa2.csa2_block_max(dev(s), bmax, n_visible=dev(nv))
    _sync_ok(csa2)
    for b in range(B):
        ref = np.full(bmax.shape[1], -np.inf, np.float32)
        m = oracle.block_max(s[b, :nv[b]], 8)
        ref[:m.size] = m
        assert np.array_equal(bmax[b].cpu().numpy(), ref)
    blocks = rng.integers(-1, 1200, (B, 96)).astype(np.int32)
    for lo, hi, nvl in ((0, 4096, [4096, 100, 0]), (4096, 8192, [4096, 4000, 5]), (128, 256, [128, 0, 64])):
        pool = torch.empty(B, 96 * 8, dtype=torch.int32, device="cuda")
        csa2.csa2_shard_pool(dev(blocks), lo, hi, pool, n_visible=dev(np.array(nvl, np.int32)))
        _sync_ok(csa2)
        p = blocks[:, :, None].astype(np.int64) * 8 + np.arange(8)
        ok = (blocks[:, :, None] >= 0) & (p >= lo) & (p < hi) & (p - lo < np.array(nvl)[:, None, None])
        assert np.array_equal(pool.cpu().numpy(), np.where(ok, p - lo, -1).reshape(B, -1))


def test_attention_merge_matches_oracle(csa2):
    rng = np.random.default_rng(23)
    R, nq = 3, 5
    parts = rng.standard_normal((R, nq, 64, 512)).astype(np.float32)
    lses = (rng.standard_normal((R, nq, 64)) * 4).astype(np.float32)
    lses[1, 0, :] = -np.inf                 # rank 1 holds no rows of query 0
    lses[:, 1, 3] = -np.inf                 # no rows at all for (query 1, head 3)
    out = torch.empty(nq, 64, 512, dtype=torch.bfloat16, device="cuda")
    out32 = torch.empty(nq, 64, 512, dtype=torch.float32, device="cuda")
    lse = torch.empty(nq, 64, dtype=torch.float32, device="cuda")
    csa2.csa2_attn_merge(dev(parts), dev(lses), out, out_f32=out32, lse_out=lse)
    _sync_ok(csa2)
    assert torch.equal(out, out32.to(torch.bfloat16))
    o, l = out32.cpu().numpy(), lse.cpu().numpy()
    for q in range(nq):
        ref, ref_l = oracle.attn_merge(parts[:, q].astype(np.float64), lses[:, q].astype(np.float64))
        np.testing.assert_allclose(o[q], ref, rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(l[q], ref_l, rtol=1e-6, atol=1e-6)
    assert np.all(o[1, 3] == 0) and l[1, 3] == -np.inf


def _unsharded(csa2, g, case, k, pool_blocks=0):
    B = case.B
    idx = torch.empty(B, k, dtype=torch.int32, device="cuda")
    if pool_blocks:
        pool = torch.empty(B, pool_blocks * 8, dtype=torch.int32, device="cuda")
        full = torch.empty(B, k, dtype=torch.int32, device="cuda")
        csa2.csa2_index_topk(g["q_data"], g["q_e8m0"], g["w"], g["ik_data"], g["ik_scale"], g["n_visible"], k, full,
                             csa2.index_topk_workspace(B, case.cap, k, pool_blocks), pool_blocks=pool_blocks,
                             pool=pool)
        csa2.csa2_index_topk(g["q_re_data"], g["q_re_e8m0"], g["w_re"], g["ik_data"], g["ik_scale"],
                             g["n_visible"], k, idx, csa2.index_topk_workspace(B, pool_blocks * 8, k),
                             positions=pool)
    else:
        full = idx
        csa2.csa2_index_topk(g["q_data"], g["q_e8m0"], g["w"], g["ik_data"], g["ik_scale"], g["n_visible"], k, idx,
                             csa2.index_topk_workspace(B, case.cap, k))
    out = torch.empty(B, case.L, 64, 512, dtype=torch.bfloat16, device="cuda")
    out32 = torch.empty(B, case.L, 64, 512, dtype=torch.float32, device="cuda")
    csa2.csa2_sparse_attn_decode(g["Q"], g["kv_data"], g["kv_scale"], g["n_visible"], idx, g["swa"], out,
                                 csa2.attn_workspace(B * case.L, k, case.n_swa), out_f32=out32)
    _sync_ok(csa2)
    return idx, full, out32


def _to_dev(a):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.to(torch.bfloat16) if t.dtype == torch.float32 and t.dim() == 4 else t


@pytest.mark.parametrize("world", [2, 3, 4])
def test_sharded_decode_step_equals_unsharded_and_oracle(csa2, world):
    case = DecodeCase(workload=99, Ns=[65536, 40000, 1000], L=2)
    g = case.to_device()
    k = 512
    ref_idx, _, ref32 = _unsharded(csa2, g, case, k)
    plan = ShardPlan(case.cap, world)
    xs = [shard_inputs(case, plan, r, to=_to_dev) for r in range(world)]
    idx, out, out32, lse = sequential_decode_step(Csa2Ops("cuda"), plan, xs, k=k)
    _sync_ok(csa2)
    assert torch.equal(idx, ref_idx)                 # same scores, same deterministic selection
    assert torch.equal(out, out32.to(torch.bfloat16))
    assert attn_row_error(out32.cpu().numpy(), ref32.cpu().numpy()) <= SHARD_ROW_TOL
    gi, o32 = idx.cpu().numpy(), out32.cpu().numpy()
    for b in range(case.B):
        check_topk(case.oracle_scores(b), gi[b], k)
        for l in range(case.L):
            ref, _ = case.oracle_attention(b, l, gi[b])
            assert attn_row_error(o32[b, l], ref) <= ATTN_ROW_TOL


def test_sharded_decode_step_with_pool_equals_unsharded(csa2):
    case = DecodeCase(workload=100, Ns=[131072, 70000], reindex=True, planted_blocks=64)
    g = case.to_device()
    k, nblk = 512, 2048
    ref_idx, ref_full, ref32 = _unsharded(csa2, g, case, k, pool_blocks=nblk)
    plan = ShardPlan(case.cap, 3)
    xs = [shard_inputs(case, plan, r, to=_to_dev, reindex=True) for r in range(3)]
    idx, out, out32, lse, idx_full = sequential_decode_step(Csa2Ops("cuda"), plan, xs, k=k, pool_blocks=nblk)
    _sync_ok(csa2)
    assert torch.equal(idx_full, ref_full)
    assert torch.equal(idx, ref_idx)
    assert attn_row_error(out32.cpu().numpy(), ref32.cpu().numpy()) <= SHARD_ROW_TOL
    gi, o32 = idx.cpu().numpy(), out32.cpu().numpy()
    for b in range(case.B):
        ref, _ = case.oracle_attention(b, 0, gi[b])
        assert attn_row_error(o32[b, 0], ref) <= ATTN_ROW_TOL
