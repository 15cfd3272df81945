"""Context sharding of the decode step: a sequence's entries split into
contiguous ranges, one per rank.

"DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", section
2.3 (the indexer's Top-K over all visible entries; one softmax over the
selected rows and the layer's SWA window) and section 2.3.2 (the block pool
ranked by block maxima). Both stay exact when the entries are split:

* a global Top-K winner beats every entry of its own range, so it is in that
  range's local Top-K; one all-gather of each rank's (score, position)
  candidates and a Top-K over them reproduce the global selection (blocks of
  the pool likewise, ranked by their maxima);
* attention over the union of disjoint row sets is the log-sum-exp merge of
  each set's normalised output, so each rank attends to the selected rows it
  holds (the last rank also to the SWA rows) and one all-gather of the
  partial outputs and their lse lets every rank merge in rank order.

A step has two exchange points (three with the pool). `ShardPlan` holds the
ranges; `decode_step` runs one rank's side over a communicator (an
all-gather); `sequential_decode_step` runs every rank's side on one device
in turn, with the all-gather replaced by stacking. Both call the same phase
functions against an `ops` object: `Csa2Ops` (the CUDA library) here, a CPU
implementation in the tests.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

BLOCK = 8     # positions per pool block (section 2.3.2)
TOPK = 512    # selected entries per query


@dataclass(frozen=True)
class ShardPlan:
    """Ranges [lo_r, hi_r) of a capacity `cap` split over `world` ranks. Every
    bound but the last is a multiple of `align` (a multiple of the pool block,
    so no block straddles two ranks)."""

    cap: int
    world: int
    align: int = 128

    def __post_init__(self):
        if self.world < 1 or self.cap < 0 or self.align % BLOCK:
            raise ValueError("bad shard plan")

    def bounds(self, rank: int) -> tuple[int, int]:
        units = -(-self.cap // self.align)
        per = -(-units // self.world)
        lo = min(rank * per * self.align, self.cap)
        hi = min((rank + 1) * per * self.align, self.cap)
        return lo, hi

    def all_bounds(self) -> list[tuple[int, int]]:
        return [self.bounds(r) for r in range(self.world)]

    def local_visible(self, rank: int, n_visible):
        """Per-sequence visible count inside the rank's range (set up once with
        the caches; a rank's appends advance it)."""
        lo, hi = self.bounds(rank)
        return [max(0, min(int(n), hi) - lo) for n in n_visible]

    def swa_owner(self) -> int:
        """The rank that attends to the SWA rows: the one holding the tail."""
        return self.world - 1


@dataclass
class ShardInputs:
    """One rank's inputs to a decode step. The planes hold the rank's entries
    at local positions; n_visible counts the visible ones among them."""

    q_data: object
    q_e8m0: object
    w: object
    ik_data: object
    ik_scale: object
    kv_data: object
    kv_scale: object
    n_visible: object
    Q: object
    swa: object            # [B, L, n_swa, 512] on the SWA owner, None elsewhere
    q_re: tuple | None = None   # (q_data, q_e8m0, w) of the re-indexing layer with the pool


# ------------------------------------------------------------------ phase functions

def phase_candidates(ops, x: ShardInputs, lo: int, k: int, pool_blocks: int = 0):
    """Local scan and Top-k of one rank; returns the candidates to all-gather
    (and, with the pool, the block candidates and the rank's scores)."""
    scores = ops.score(x.q_data, x.q_e8m0, x.w, x.ik_data, x.ik_scale, x.n_visible)
    cols = ops.topk(scores, k, x.n_visible)
    cand = ops.candidates(scores, cols, lo)
    if not pool_blocks:
        return cand, None, scores
    bmax = ops.block_max(scores, x.n_visible)
    bcols = ops.topk(bmax, pool_blocks, None)
    bcand = ops.candidates(bmax, bcols, lo // BLOCK)
    return cand, bcand, scores


def phase_reindex(ops, x: ShardInputs, blocks, lo: int, hi: int, k: int):
    """Re-score the merged pool's positions in the rank's range with the
    re-indexing layer's query; returns its candidates."""
    pos = ops.shard_pool(blocks, lo, hi, x.n_visible)
    q_data, q_e8m0, w = x.q_re
    s = ops.score(q_data, q_e8m0, w, x.ik_data, x.ik_scale, x.n_visible, positions=pos)
    cols = ops.topk(s, k, None)
    return ops.candidates(s, cols, lo, positions=pos)


def phase_attention(ops, x: ShardInputs, idx, lo: int, hi: int):
    """Attention of the rank's share of the selected rows (plus the SWA rows
    on their owner): normalised partial outputs and their lse."""
    local = ops.shard_positions(idx, lo, hi)
    return ops.attn(x.Q, x.kv_data, x.kv_scale, x.n_visible, local, x.swa)


# ------------------------------------------------------------------ drivers

def decode_step(ops, comm, plan: ShardPlan, rank: int, x: ShardInputs, k: int = TOPK, pool_blocks: int = 0):
    """One rank's side of a context-sharded decode step. `comm.all_gather(t)`
    returns the rank-ordered stack [world, *t.shape]. Returns (idx [B,k]
    global positions, out, out_f32, lse); with the pool, idx comes from the
    re-indexing layer and the indexing layer's own Top-k is returned as well."""
    lo, hi = plan.bounds(rank)
    cand, bcand, _ = phase_candidates(ops, x, lo, k, pool_blocks)
    idx_full = ops.merge(comm.all_gather(cand), k)
    idx = idx_full
    if pool_blocks:
        blocks = ops.merge(comm.all_gather(bcand), pool_blocks)
        idx = ops.merge(comm.all_gather(phase_reindex(ops, x, blocks, lo, hi, k)), k)
    o32, lse = phase_attention(ops, x, idx, lo, hi)
    out, out32, lse_all = ops.attn_merge(comm.all_gather(o32), comm.all_gather(lse))
    return (idx, out, out32, lse_all) + ((idx_full,) if pool_blocks else ())


def sequential_decode_step(ops, plan: ShardPlan, xs: list[ShardInputs], k: int = TOPK, pool_blocks: int = 0):
    """Every rank's side run in turn on one device; each exchange is the stack
    of the ranks' tensors in rank order. Same result as `decode_step` on
    `plan.world` ranks."""
    stack = ops.stack
    bounds = plan.all_bounds()
    phase = [phase_candidates(ops, x, lo, k, pool_blocks) for x, (lo, _) in zip(xs, bounds)]
    idx_full = ops.merge(stack([c for c, _, _ in phase]), k)
    idx = idx_full
    if pool_blocks:
        blocks = ops.merge(stack([b for _, b, _ in phase]), pool_blocks)
        idx = ops.merge(stack([phase_reindex(ops, x, blocks, lo, hi, k) for x, (lo, hi) in zip(xs, bounds)]), k)
    parts = [phase_attention(ops, x, idx, lo, hi) for x, (lo, hi) in zip(xs, bounds)]
    out, out32, lse_all = ops.attn_merge(stack([p[0] for p in parts]), stack([p[1] for p in parts]))
    return (idx, out, out32, lse_all) + ((idx_full,) if pool_blocks else ())


# ------------------------------------------------------------------ CUDA ops

class Csa2Ops:
    """The phase steps on the CUDA library (device tensors, current stream)."""

    def __init__(self, device, sm_scale: float = 1.0):
        from . import csa2
        self.csa2 = csa2
        self.device = torch.device(device)
        self.sm_scale = sm_scale

    def _i32(self, *shape):
        return torch.empty(*shape, dtype=torch.int32, device=self.device)

    def score(self, q_data, q_e8m0, w, ik_data, ik_scale, n_visible, positions=None):
        B = ik_data.shape[0]
        n = positions.shape[1] if positions is not None else ik_data.shape[1]
        s = torch.empty(B, n, dtype=torch.float32, device=self.device)
        self.csa2.csa2_index_score(q_data, q_e8m0, w, ik_data, ik_scale, n_visible, s, positions=positions)
        return s

    def topk(self, scores, k, n_valid):
        B, n = scores.shape
        idx = self._i32(B, k)
        self.csa2.csa2_topk(scores, k, idx, self.csa2.topk_workspace(B, n, k, self.device), n_valid=n_valid)
        return idx

    def candidates(self, scores, cols, offset, positions=None):
        cand = self._i32(cols.shape[0], cols.shape[1], 2)
        self.csa2.csa2_topk_candidates(scores, cols, offset, cand, positions=positions)
        return cand

    def block_max(self, scores, n_visible):
        B, n = scores.shape
        bmax = torch.empty(B, -(-n // BLOCK), dtype=torch.float32, device=self.device)
        self.csa2.csa2_block_max(scores, bmax, n_visible=n_visible)
        return bmax

    def merge(self, cand, k_out):
        R, B, k = cand.shape[0], cand.shape[1], cand.shape[2]
        idx = self._i32(B, k_out)
        self.csa2.csa2_topk_merge(cand, k_out, idx, self.csa2.merge_workspace(R, B, k, k_out, self.device))
        return idx

    def shard_positions(self, idx, lo, hi):
        local = torch.empty_like(idx)
        self.csa2.csa2_shard_positions(idx, lo, hi, local)
        return local

    def shard_pool(self, blocks, lo, hi, n_visible):
        pool = self._i32(blocks.shape[0], blocks.shape[1] * BLOCK)
        self.csa2.csa2_shard_pool(blocks, lo, hi, pool, n_visible=n_visible)
        return pool

    def attn(self, Q, kv_data, kv_scale, n_visible, idx, swa):
        B, L = Q.shape[0], Q.shape[1]
        out = torch.empty_like(Q)
        o32 = torch.empty(Q.shape, dtype=torch.float32, device=self.device)
        lse = torch.empty(B, L, self.csa2.HEADS, dtype=torch.float32, device=self.device)
        n_swa = swa.shape[2] if swa is not None else 0
        ws = self.csa2.attn_workspace(B * L, idx.shape[1], n_swa, self.device)
        self.csa2.csa2_sparse_attn_decode(Q, kv_data, kv_scale, n_visible, idx, swa, out, ws, out_f32=o32, lse=lse,
                                     sm_scale=self.sm_scale)
        return o32, lse

    def attn_merge(self, parts, lses):
        out = torch.empty(parts.shape[1:], dtype=torch.bfloat16, device=self.device)
        out32 = torch.empty(parts.shape[1:], dtype=torch.float32, device=self.device)
        lse = torch.empty(lses.shape[1:], dtype=torch.float32, device=self.device)
        self.csa2.csa2_attn_merge(parts, lses, out, out_f32=out32, lse_out=lse)
        return out, out32, lse

    @staticmethod
    def stack(ts):
        return torch.stack(ts)


class TorchComm:
    """All-gather over torch.distributed (NCCL for device tensors, gloo for
    host tensors)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.world = dist.get_world_size(group)

    def all_gather(self, t):
        t = t.contiguous()
        if t.is_cuda:
            out = torch.empty((self.world,) + tuple(t.shape), dtype=t.dtype, device=t.device)
            self.dist.all_gather_into_tensor(out, t, group=self.group)
            return out
        parts = [torch.empty_like(t) for _ in range(self.world)]
        self.dist.all_gather(parts, t, group=self.group)
        return torch.stack(parts)
