"""Shared helpers of the GPU parity tests: oracle-built caches and the
comparison rules.

Comparison rules (the tolerances are derived in the design notes):
  - packing and dequantised bytes: bit-exact;
  - Top-K: the GPU and oracle index sets are equal except for positions whose
    oracle fp32 score lies within 1e-5 relative of the oracle's K-th score;
  - attention (given the oracle's index set): max over (query, head) rows of
    max_c |o_gpu - o_ref| / max_c |o_ref| <= 2e-3 for the fp32-accumulated
    output; the bf16 output is the round-to-nearest-even of the fp32 output.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from fp4_kv_cache_02_gb300.inputs import CAP_ALIGN, decode_sequence, round_up

TOPK_REL_TOL = 1e-5
ATTN_ROW_TOL = 2e-3


def dev(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def check_topk(ref_scores32, got_idx, k, positions=None, ref_idx=None):
    """Top-K rule against the oracle; ref_scores32 are oracle fp32 scores over the
    candidates (aligned with `positions` if given). Returns #boundary swaps."""
    got = [int(p) for p in got_idx if p >= 0]
    assert len(got) == len(set(got)), "duplicate positions"
    assert list(got_idx[:len(got)]) == sorted(got), "GPU indices must be ascending, -1 padded"
    if ref_idx is None:
        ref_idx, _ = oracle.topk(ref_scores32, k, positions=positions)
    ref = [int(p) for p in ref_idx if p >= 0]
    assert len(got) == len(ref), (len(got), len(ref))
    if not ref:
        return 0
    pos = np.arange(len(ref_scores32)) if positions is None else np.asarray(positions)
    score_of = {int(p): float(s) for p, s in zip(pos, ref_scores32) if p >= 0}
    kth = score_of[ref[-1]]  # oracle order is (score desc, position asc)
    diff = set(got) ^ set(ref)
    for p in diff:
        assert abs(score_of[p] - kth) <= TOPK_REL_TOL * abs(kth), (p, score_of[p], kth)
    return len(diff) // 2


def attn_row_error(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max(axis=-1)
    num = np.abs(got - ref).max(axis=-1)
    den = np.where(den == 0, 1.0, den)
    return float((num / den).max())


def bf16_of(x_f32: torch.Tensor) -> torch.Tensor:
    return x_f32.to(torch.bfloat16)


class DecodeCase:
    """B sequences of oracle-quantised caches with capacity cap >= max(N)."""

    def __init__(self, workload, Ns, L=1, n_swa=128, reindex=False, planted_blocks=0, garbage_tail=True,
                 gen_device=None):
        self.B = len(Ns)
        self.Ns = list(Ns)
        self.cap = round_up(max(max(Ns), 1), CAP_ALIGN)
        self.L = L
        self.n_swa = n_swa
        B, cap = self.B, self.cap
        rng = np.random.default_rng(12345)
        self.ik_data = np.zeros((B, cap, 64), np.uint8)
        self.ik_scale = np.zeros((B, cap, 4), np.uint8)
        self.kv_data = np.zeros((B, cap, 256), np.uint8)
        self.kv_scale = np.zeros((B, cap, 32), np.uint8)
        if garbage_tail:
            # bytes past n_visible are arbitrary (NaN scales included) and must never matter
            for b, N in enumerate(Ns):
                for plane in (self.ik_data, self.ik_scale, self.kv_data, self.kv_scale):
                    plane[b, N:] = rng.integers(0, 256, plane[b, N:].shape, dtype=np.uint8)
        self.q_idx = np.zeros((B, 32, 128), np.float32)
        self.q_data = np.zeros((B, 32, 64), np.uint8)
        self.q_e8m0 = np.zeros((B, 32, 4), np.uint8)
        self.w = np.zeros((B, 32), np.float32)
        self.Q = np.zeros((B, L, 64, 512), np.float32)
        self.swa = np.zeros((B, L, n_swa, 512), np.uint8)
        if reindex:
            self.q_re = np.zeros((B, 32, 128), np.float32)
            self.q_re_data = np.zeros((B, 32, 64), np.uint8)
            self.q_re_e8m0 = np.zeros((B, 32, 4), np.uint8)
            self.w_re = np.zeros((B, 32), np.float32)
        self.planted = []
        for b, N in enumerate(Ns):
            d = decode_sequence(workload, b, N, L=L, reindex=reindex, planted_blocks=planted_blocks, n_swa=n_swa,
                                device=gen_device)
            self.q_idx[b] = d["q_idx"]
            self.q_data[b], self.q_e8m0[b] = oracle.quant_mxfp4(d["q_idx"])
            self.w[b] = d["w"]
            if N:
                self.ik_data[b, :N], self.ik_scale[b, :N] = oracle.quant_mxfp4(d["ik"])
                self.kv_data[b, :N], self.kv_scale[b, :N] = oracle.pack_kv_fp4(d["kv"])
            self.Q[b] = d["Q"]
            if n_swa:
                self.swa[b] = oracle.pack_fp8(d["swa"].reshape(-1)).reshape(L, n_swa, 512)
            if reindex:
                self.q_re[b] = d["q_re"]
                self.q_re_data[b], self.q_re_e8m0[b] = oracle.quant_mxfp4(d["q_re"])
                self.w_re[b] = d["w_re"]
            if planted_blocks:
                self.planted.append(d["planted"])
        self.n_visible = np.array(Ns, np.int32)

    def to_device(self, device="cuda"):
        g = {}
        for name in ("ik_data", "ik_scale", "kv_data", "kv_scale", "q_data", "q_e8m0", "w", "swa", "n_visible"):
            g[name] = dev(getattr(self, name), device)
        g["Q"] = dev(self.Q, device).to(torch.bfloat16)
        g["q_idx"] = dev(self.q_idx, device).to(torch.bfloat16)
        if hasattr(self, "q_re"):
            g["q_re"] = dev(self.q_re, device).to(torch.bfloat16)
            g["q_re_data"] = dev(self.q_re_data, device)
            g["q_re_e8m0"] = dev(self.q_re_e8m0, device)
            g["w_re"] = dev(self.w_re, device)
        return g

    def oracle_scores(self, b, q="full"):
        if q == "full":
            qd, qs, w = self.q_data[b], self.q_e8m0[b], self.w[b]
        else:
            qd, qs, w = self.q_re_data[b], self.q_re_e8m0[b], self.w_re[b]
        return oracle.index_score(qd, qs, w, self.ik_data[b], self.ik_scale[b], n=self.Ns[b])[0]

    def oracle_attention(self, b, l, idx):
        return oracle.sparse_attn(self.Q[b, l], self.kv_data[b], self.kv_scale[b], idx, self.swa[b, l])
