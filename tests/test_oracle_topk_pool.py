"""Pins of the oracle's Top-K and hierarchical block pool: brute force on tiny
inputs with planted ties, and the invariants the report's construction
implies (a pool covering every block reproduces the full scan; the Full
layer's Top-512 lies inside its pool)."""

import numpy as np
import pytest

from fp4_kv_cache_02_gb300.inputs import bf16_round


def _brute_topk(scores, k, positions=None):
    n = len(scores)
    pos = list(range(n)) if positions is None else list(positions)
    items = [(-float(s), int(p)) for s, p in zip(scores, pos) if p >= 0 and np.isfinite(s)]
    items.sort()
    out = [p for _, p in items[:k]]
    return out + [-1] * (k - len(out))


@pytest.mark.parametrize("n,k", [(1, 1), (7, 3), (16, 16), (40, 8), (64, 64), (64, 100), (0, 4)])
def test_topk_brute_force_with_ties(orc, n, k):
    rng = np.random.default_rng(100 + n + k)
    s = rng.integers(0, 5, n).astype(np.float32)  # many ties
    idx, nv = orc.topk(s, k)
    assert list(idx) == _brute_topk(s, k)
    assert nv == min(n, k)


def test_topk_positions_map_and_masking(orc):
    rng = np.random.default_rng(7)
    s = rng.standard_normal(50).astype(np.float32)
    pos = rng.permutation(1000)[:50].astype(np.int32)
    pos[3] = -1
    s[9] = -np.inf
    idx, nv = orc.topk(s, 20, positions=pos)
    assert list(idx) == _brute_topk(s, 20, pos)
    assert -1 not in list(idx)
    idx, nv = orc.topk(s, 60, positions=pos)
    assert nv == 48 and list(idx[48:]) == [-1] * 12


def _brute_pool(scores, block, n_blocks):
    n = len(scores)
    nb = (n + block - 1) // block
    bmax = [max(scores[b * block:min(n, (b + 1) * block)]) for b in range(nb)]
    order = sorted(range(nb), key=lambda b: (-bmax[b], b))[:n_blocks]
    kept = sorted(order)
    pool = []
    for j in range(n_blocks):
        for r in range(block):
            p = kept[j] * block + r if j < len(kept) else -1
            pool.append(p if 0 <= p < n else -1)
    return pool


@pytest.mark.parametrize("n,block,nbk", [(61, 8, 4), (64, 8, 8), (100, 8, 20), (33, 4, 3), (5, 8, 2)])
def test_pool_brute_force(orc, n, block, nbk):
    rng = np.random.default_rng(n * 7 + nbk)
    s = rng.integers(0, 6, n).astype(np.float32)
    pool, kept = orc.block_pool(s, block, nbk)
    assert list(pool) == _brute_pool(list(s), block, nbk)


@pytest.fixture(scope="module")
def scored_seq(orc):
    rng = np.random.default_rng(31)
    n = 20000
    q = bf16_round(rng.standard_normal((32, 128)).astype(np.float32))
    q2 = bf16_round(rng.standard_normal((32, 128)).astype(np.float32))
    w = rng.uniform(0, 1, 32).astype(np.float32)
    w2 = rng.uniform(0, 1, 32).astype(np.float32)
    k = bf16_round(rng.standard_normal((n, 128)).astype(np.float32))
    qd, qs = orc.quant_mxfp4(q)
    q2d, q2s = orc.quant_mxfp4(q2)
    kd, ks = orc.quant_mxfp4(k)
    s, _, _ = orc.index_score(qd, qs, w, kd, ks)
    return dict(n=n, s=s, kd=kd, ks=ks, q2d=q2d, q2s=q2s, w2=w2)


def test_full_topk_lies_inside_the_pool(orc, scored_seq):
    s = scored_seq["s"]
    idx, _ = orc.topk(s, 512)
    pool, kept = orc.block_pool(s, 8, 512)  # even a 512-block pool holds the Top-512
    assert set(idx.tolist()) <= set(pool.tolist())
    pool, kept = orc.block_pool(s, 8, 2048)
    assert kept == 2048
    assert set(idx.tolist()) <= set(pool.tolist())


def test_pool_covering_every_block_reproduces_the_full_scan(orc, scored_seq):
    c = scored_seq
    n = 16000  # ceil(n/8) = 2000 <= 2048 blocks: every block is in the pool
    s = c["s"][:n]
    pool, kept = orc.block_pool(s, 8, 2048)
    assert kept == 2000
    assert sorted(p for p in pool if p >= 0) == list(range(n))
    full, _, _ = orc.index_score(c["q2d"], c["q2s"], c["w2"], c["kd"], c["ks"], n=n)
    pooled, _, _ = orc.index_score(c["q2d"], c["q2s"], c["w2"], c["kd"], c["ks"], positions=pool)
    a, _ = orc.topk(full, 512)
    b, _ = orc.topk(pooled, 512, positions=pool)
    assert list(a) == list(b)
