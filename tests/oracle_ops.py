"""The context-sharding phase steps on the CPU oracle (torch CPU tensors in
and out, so that gloo ranks can all-gather them). Used by the CPU tests of
the sharding host logic; the oracle does the arithmetic, numpy only moves
data and applies the masks that the C ABI defines."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from fp4_kv_cache_02_gb300.sharding import BLOCK, ShardInputs, ShardPlan


def _np(t):
    return t.numpy() if isinstance(t, torch.Tensor) else np.asarray(t)


def _ascending(idx, k):
    got = np.sort(idx[idx >= 0])
    return np.concatenate([got, -np.ones(k - got.size, np.int32)]).astype(np.int32)


class OracleOps:
    def score(self, q_data, q_e8m0, w, ik_data, ik_scale, n_visible, positions=None):
        q_data, q_e8m0, w, ik_data, ik_scale, nv = map(_np, (q_data, q_e8m0, w, ik_data, ik_scale, n_visible))
        B = ik_data.shape[0]
        n = positions.shape[1] if positions is not None else ik_data.shape[1]
        out = np.full((B, n), -np.inf, np.float32)
        for b in range(B):
            if positions is None:
                if nv[b]:
                    out[b, :nv[b]] = oracle.index_score(q_data[b], q_e8m0[b], w[b], ik_data[b], ik_scale[b],
                                                        n=int(nv[b]))[0]
            else:
                p = _np(positions)[b].copy()
                p[p >= nv[b]] = -1
                out[b] = oracle.index_score(q_data[b], q_e8m0[b], w[b], ik_data[b], ik_scale[b], positions=p)[0]
        return torch.from_numpy(out)

    def topk(self, scores, k, n_valid):
        s = _np(scores)
        idx = np.zeros((s.shape[0], k), np.int32)
        for b in range(s.shape[0]):
            row = s[b].copy()
            if n_valid is not None:
                row[int(_np(n_valid)[b]):] = -np.inf
            idx[b] = _ascending(oracle.topk(row, k)[0], k)
        return torch.from_numpy(idx)

    def candidates(self, scores, cols, offset, positions=None):
        s, c = _np(scores), _np(cols)
        B, k = c.shape
        vals = np.full((B, k), -np.inf, np.float32)
        pos = np.full((B, k), -1, np.int32)
        for b in range(B):
            for j in range(k):
                col = int(c[b, j])
                if 0 <= col < s.shape[1]:
                    p = int(_np(positions)[b, col]) if positions is not None else col
                    if p >= 0:
                        vals[b, j] = s[b, col]
                        pos[b, j] = p + offset
        return torch.from_numpy(np.stack([vals.view(np.int32), pos], -1))

    def block_max(self, scores, n_visible):
        s, nv = _np(scores), _np(n_visible)
        nb = -(-s.shape[1] // BLOCK)
        out = np.full((s.shape[0], nb), -np.inf, np.float32)
        for b in range(s.shape[0]):
            m = oracle.block_max(s[b, :int(nv[b])], BLOCK)
            out[b, :m.size] = m
        return torch.from_numpy(out)

    def merge(self, cand, k_out):
        c = _np(cand)
        R, B, k, _ = c.shape
        idx = np.zeros((B, k_out), np.int32)
        for b in range(B):
            vals = np.ascontiguousarray(c[:, b, :, 0]).view(np.float32).reshape(-1)
            pos = np.ascontiguousarray(c[:, b, :, 1]).reshape(-1)
            idx[b] = _ascending(oracle.topk(vals, k_out, positions=pos)[0], k_out)
        return torch.from_numpy(idx)

    def shard_positions(self, idx, lo, hi):
        i = _np(idx)
        return torch.from_numpy(np.where((i >= lo) & (i < hi), i - lo, -1).astype(np.int32))

    def shard_pool(self, blocks, lo, hi, n_visible):
        bl, nv = _np(blocks), _np(n_visible)
        B, nb = bl.shape
        p = bl[:, :, None].astype(np.int64) * BLOCK + np.arange(BLOCK)[None, None, :]
        ok = (bl[:, :, None] >= 0) & (p >= lo) & (p < hi) & (p - lo < nv[:, None, None])
        return torch.from_numpy(np.where(ok, p - lo, -1).reshape(B, nb * BLOCK).astype(np.int32))

    def attn(self, Q, kv_data, kv_scale, n_visible, idx, swa):
        Q, kvd, kvs, i = map(_np, (Q, kv_data, kv_scale, idx))
        B, L, H, D = Q.shape
        out = np.zeros((B, L, H, D), np.float64)
        lse = np.zeros((B, L, H), np.float64)
        for b in range(B):
            for l in range(L):
                out[b, l], lse[b, l] = oracle.sparse_attn(Q[b, l], kvd[b], kvs[b], i[b],
                                                          None if swa is None else _np(swa)[b, l])
        return torch.from_numpy(out), torch.from_numpy(lse)

    def attn_merge(self, parts, lses):
        P, S = _np(parts), _np(lses)
        _, B, L, H, D = P.shape
        out = np.zeros((B, L, H, D), np.float64)
        lse = np.zeros((B, L, H), np.float64)
        for b in range(B):
            for l in range(L):
                out[b, l], lse[b, l] = oracle.attn_merge(P[:, b, l], S[:, b, l])
        o = torch.from_numpy(out)
        return o, o, torch.from_numpy(lse)

    @staticmethod
    def stack(ts):
        return torch.stack(ts)


def shard_inputs(case, plan: ShardPlan, rank: int, to=None, reindex=False):
    """Rank `rank`'s share of a tests.helpers.DecodeCase: the planes of its
    range, its local visible counts, the SWA rows on their owner. `to` maps a
    numpy array to the tensor type the ops take (CPU torch by default)."""
    to = to or (lambda a: torch.from_numpy(np.ascontiguousarray(a)))
    lo, hi = plan.bounds(rank)
    nv = np.array(plan.local_visible(rank, case.Ns), np.int32)
    q_re = None
    if reindex:
        q_re = (to(case.q_re_data), to(case.q_re_e8m0), to(case.w_re))
    return ShardInputs(
        q_data=to(case.q_data), q_e8m0=to(case.q_e8m0), w=to(case.w),
        ik_data=to(case.ik_data[:, lo:hi]), ik_scale=to(case.ik_scale[:, lo:hi]),
        kv_data=to(case.kv_data[:, lo:hi]), kv_scale=to(case.kv_scale[:, lo:hi]),
        n_visible=to(nv), Q=to(case.Q), swa=to(case.swa) if rank == plan.swa_owner() else None, q_re=q_re)


def unsharded_reference(case, k, pool_blocks=0):
    """The whole step on the oracle without sharding: (idx ascending [B,k],
    out [B,L,H,D], idx of the indexing layer)."""
    B = case.B
    idx = np.zeros((B, k), np.int32)
    idx_full = np.zeros((B, k), np.int32)
    out = np.zeros(case.Q.shape, np.float64)
    for b in range(B):
        s = case.oracle_scores(b)
        idx_full[b] = _ascending(oracle.topk(s, k)[0], k)
        if pool_blocks:
            pool, _ = oracle.block_pool(s, BLOCK, pool_blocks)
            s2 = oracle.index_score(case.q_re_data[b], case.q_re_e8m0[b], case.w_re[b], case.ik_data[b],
                                    case.ik_scale[b], positions=pool)[0]
            idx[b] = _ascending(oracle.topk(s2, k, positions=pool)[0], k)
        else:
            idx[b] = idx_full[b]
        for l in range(case.L):
            out[b, l] = case.oracle_attention(b, l, idx[b])[0]
    return idx, out, idx_full
