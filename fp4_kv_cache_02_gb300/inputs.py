"""Seeded synthetic inputs shaped like the workloads of the CSA2 decode and
prefill hot path.

This module only draws random numbers and rounds them to bf16 (the input
type of the product path). It holds none of the method's arithmetic: no
quantisation, scoring, selection or attention. Both the CPU oracle (through
the tests) and the CUDA path consume what it produces.

Workloads (sizes from the decoder setup in "DeepSeek-V4.1-Flash: Pushing the
Limits of KV Cache Compression": 32 indexer heads x 128, 64 attention heads x
512, Top-K 512, SWA window 128, pool of 2,048 blocks x 8):

  0  decode, 1 sequence, N = 4,096 visible entries
  1  Full-layer decode, 32 sequences, N = 65,536 each
  2  Reindex-layer decode with the block pool, 8 sequences, N = 1,048,576,
     64 planted high-affinity blocks per sequence
  3  prefill chunk, 4,096 causal queries after 126,976 cached entries
  4  long-context decode, 4 sequences, N = 1,048,576, 1 Full + 3 Reuse layers

Value distributions: indexer q, keys, latents and SWA rows ~ N(0,1); head
weights ~ U(0,1); main Q ~ N(0,1)/sqrt(512). Seeds: workload 0 uses 0,
workload 1 uses the sequence id, the others 1000 * workload + sequence.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

IDX_HEADS = 32
IDX_DIM = 128
HEADS = 64
HEAD_DIM = 512
TOPK = 512
SWA_W = 128
POOL_BLOCK = 8
POOL_BLOCKS = 2048
CAP_ALIGN = 128  # plane capacity is a multiple of this many entries


@dataclass(frozen=True)
class Workload:
    id: int
    name: str
    kind: str          # "decode", "reindex" or "prefill"
    B: int             # sequences (decode) or 1 (prefill)
    N: int             # visible entries per sequence (prefill: total after the chunk)
    L: int = 1         # layers sharing the indices (1 Full + L-1 Reuse)
    T: int = 0         # prefill queries
    planted_blocks: int = 0


WORKLOADS = {
    0: Workload(0, "decode_b1_n4096", "decode", 1, 4096),
    1: Workload(1, "full_decode_b32_n65536", "decode", 32, 65536),
    2: Workload(2, "reindex_decode_b8_n1048576_pool2048x8", "reindex", 8, 1 << 20,
                planted_blocks=64),
    3: Workload(3, "prefill_t4096_after_126976", "prefill", 1, 131072, T=4096),
    4: Workload(4, "long_decode_b4_n1048576_full_plus_3_reuse", "decode", 4, 1 << 20, L=4),
}


def seed_for(workload: int, seq: int) -> int:
    if workload == 0:
        return 0
    if workload == 1:
        return seq
    return 1000 * workload + seq


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float values to the nearest bf16 and return them as float32."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def _normal(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32)


def _big_normal(rng: np.random.Generator, shape, seed: int, device) -> np.ndarray:
    """N(0,1) float32 on the host; drawn with torch's seeded generator on
    `device` when given (fast for the 1M-entry workloads), else with numpy."""
    if device is None:
        return _normal(rng, shape)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).cpu().numpy()


def decode_sequence(workload: int, seq: int, N: int, L: int = 1,
                    reindex: bool = False, planted_blocks: int = 0,
                    n_swa: int = SWA_W, device=None) -> dict:
    """Host (numpy float32, bf16-exact) inputs of one decode sequence.

    Keys: q_idx [32,128], w [32], ik [N,128], kv [N,512], Q [L,64,512],
    swa [L,n_swa,512]; for reindex also q_re [32,128], w_re [32], and
    planted (the planted block ids, sorted). With `device`, the two large
    planes (ik, kv) are drawn by torch's generator on that device."""
    seed = seed_for(workload, seq)
    rng = np.random.default_rng(seed)
    out = {}
    out["q_idx"] = bf16_round(_normal(rng, (IDX_HEADS, IDX_DIM)))
    out["w"] = rng.uniform(0.0, 1.0, IDX_HEADS).astype(np.float32)
    ik = _big_normal(rng, (N, IDX_DIM), 4 * seed + 1, device)
    out["kv"] = bf16_round(_big_normal(rng, (N, HEAD_DIM), 4 * seed + 2, device))
    out["Q"] = bf16_round(_normal(rng, (L, HEADS, HEAD_DIM)) / np.float32(math.sqrt(HEAD_DIM)))
    out["swa"] = bf16_round(_normal(rng, (L, n_swa, HEAD_DIM)))
    if reindex:
        out["q_re"] = bf16_round(_normal(rng, (IDX_HEADS, IDX_DIM)))
        out["w_re"] = rng.uniform(0.0, 1.0, IDX_HEADS).astype(np.float32)
    if planted_blocks:
        # keys aligned to u = sum_h w_h q_h of the Full layer, |u| = sqrt(128),
        # plus 0.1 * N(0,1) per channel, in blocks drawn without replacement
        u = (out["w"][:, None].astype(np.float64) * out["q_idx"].astype(np.float64)).sum(0)
        u *= math.sqrt(IDX_DIM) / np.linalg.norm(u)
        blocks = np.sort(rng.choice(N // POOL_BLOCK, planted_blocks, replace=False))
        for b in blocks:
            rows = slice(b * POOL_BLOCK, (b + 1) * POOL_BLOCK)
            ik[rows] = (u[None, :] + 0.1 * _normal(rng, (POOL_BLOCK, IDX_DIM))).astype(np.float32)
        out["planted"] = blocks.astype(np.int64)
    out["ik"] = bf16_round(ik)
    return out


def prefill_chunk(workload: int, T: int, N0: int, n_swa: int = SWA_W, device=None) -> dict:
    """Host inputs of a prefill chunk: T queries at positions N0..N0+T-1 over
    N0+T entries. Keys: q_idx [T,32,128], w [T,32], ik [N0+T,128],
    kv [N0+T,512], Q [T,64,512], swa [T+n_swa-1,512] (row r is position
    N0-(n_swa-1)+r). With `device`, the large arrays are drawn there."""
    seed = seed_for(workload, 0)
    rng = np.random.default_rng(seed)
    N = N0 + T
    return {
        "q_idx": bf16_round(_big_normal(rng, (T, IDX_HEADS, IDX_DIM), 4 * seed + 1, device)),
        "w": rng.uniform(0.0, 1.0, (T, IDX_HEADS)).astype(np.float32),
        "ik": bf16_round(_big_normal(rng, (N, IDX_DIM), 4 * seed + 2, device)),
        "kv": bf16_round(_big_normal(rng, (N, HEAD_DIM), 4 * seed + 3, device)),
        "Q": bf16_round(_big_normal(rng, (T, HEADS, HEAD_DIM), 4 * seed + 4, device)
                        / np.float32(math.sqrt(HEAD_DIM))),
        "swa": bf16_round(_normal(rng, (T + n_swa - 1, HEAD_DIM))),
    }


def device_normal(shape, seed: int, device="cuda", scale: float = 1.0) -> torch.Tensor:
    """N(0, scale^2) values rounded to bf16, drawn on the device (bench sizes)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(torch.bfloat16)


def device_uniform(shape, seed: int, device="cuda") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32)


def device_planted_keys(ik: torch.Tensor, q_idx: torch.Tensor, w: torch.Tensor, n_visible: int,
                        n_blocks: int, seed: int) -> torch.Tensor:
    """The planted high-affinity blocks of the Reindex workload, on the device:
    `n_blocks` blocks of POOL_BLOCK keys, drawn without replacement below
    `n_visible`, are overwritten in place with u + 0.1 * N(0,1) per channel,
    where u = sum_h w_h q_h scaled to norm sqrt(128) (the recipe of
    decode_sequence). ik [cap,128] bf16; returns the sorted block ids."""
    g = torch.Generator(device=ik.device)
    g.manual_seed(seed)
    u = (w.double()[:, None] * q_idx.double()).sum(0)
    u = u * (math.sqrt(IDX_DIM) / torch.linalg.vector_norm(u))
    blocks = torch.randperm(n_visible // POOL_BLOCK, generator=g, device=ik.device)[:n_blocks].sort().values
    noise = torch.randn(n_blocks, POOL_BLOCK, IDX_DIM, generator=g, device=ik.device, dtype=torch.float32)
    rows = (blocks[:, None] * POOL_BLOCK + torch.arange(POOL_BLOCK, device=ik.device)[None, :]).reshape(-1)
    ik[rows] = (u.float()[None, None, :] + 0.1 * noise).reshape(-1, IDX_DIM).to(torch.bfloat16)
    return blocks
