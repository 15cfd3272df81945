"""GPU parity of the indexer scan, Top-K, block pool and the fused index path
against the oracle, on small ragged cases and planted ties."""

import numpy as np
import pytest
import torch

import oracle

from helpers import DecodeCase, check_topk, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    from fp4_kv_cache_02_gb300 import csa2 as m
    return m


@pytest.fixture(scope="module")
def case():
    # ragged: three sequences, the longest spans several 128-entry tiles and a tail
    return DecodeCase(workload=91, Ns=[4093, 1000, 130])


def _scores_close(got, ref):
    scale = np.abs(ref[np.isfinite(ref)]).max()
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin)
    np.testing.assert_allclose(got[fin], ref[fin], rtol=1e-5, atol=1e-6 * scale)


def test_index_score_matches_oracle(csa2, case):
    g = case.to_device()
    scores = torch.empty(case.B, case.cap, dtype=torch.float32, device="cuda")
    csa2.csa2_index_score(g["q_data"], g["q_e8m0"], g["w"], g["ik_data"], g["ik_scale"], g["n_visible"], scores)
    s = scores.cpu().numpy()
    for b in range(case.B):
        ref = case.oracle_scores(b)
        _scores_close(s[b, :case.Ns[b]], ref)
        assert np.all(s[b, case.Ns[b]:] == -np.inf)


def test_index_score_with_positions(csa2, case):
    g = case.to_device()
    rng = np.random.default_rng(3)
    n_pos = 777
    pos = np.stack([rng.integers(-1, case.Ns[b] + 5, n_pos) for b in range(case.B)]).astype(np.int32)
    scores = torch.empty(case.B, n_pos, dtype=torch.float32, device="cuda")
    csa2.csa2_index_score(g["q_data"], g["q_e8m0"], g["w"], g["ik_data"], g["ik_scale"], g["n_visible"], scores,
                          positions=dev(pos))
    s = scores.cpu().numpy()
    for b in range(case.B):
        p = np.where(pos[b] < case.Ns[b], pos[b], -1).astype(np.int32)
        ref = oracle.index_score(case.q_data[b], case.q_e8m0[b], case.w[b], case.ik_data[b], case.ik_scale[b],
                                 positions=p)[0]
        _scores_close(s[b], ref)


@pytest.mark.parametrize("n,k,levels", [(1000, 512, 0), (64, 100, 5), (5000, 1, 0), (20000, 4096, 3),
                                        (3000, 512, 2), (70000, 512, 0)])
def test_topk_exact_on_identical_scores(csa2, n, k, levels):
    """Same fp32 scores in, the GPU must return exactly the oracle's set
    (ties broken by smaller position)."""
    rng = np.random.default_rng(n + k)
    B = 3
    if levels:
        s = rng.integers(0, levels, (B, n)).astype(np.float32)   # massive ties
    else:
        s = rng.standard_normal((B, n)).astype(np.float32)
    s[0, 5] = -np.inf
    s[1, 7] = np.nan
    nvalid = np.array([n, max(n // 2, 1), n - 3], np.int32)
    idx = torch.empty(B, k, dtype=torch.int32, device="cuda")
    ws = csa2.topk_workspace(B, n, k)
    csa2.csa2_topk(dev(s), k, idx, ws, n_valid=dev(nvalid))
    got = idx.cpu().numpy()
    for b in range(B):
        ref, nv = oracle.topk(s[b, :nvalid[b]], k)
        expect = sorted(int(p) for p in ref if p >= 0)
        assert list(got[b, :len(expect)]) == expect
        assert np.all(got[b, len(expect):] == -1)


@pytest.mark.parametrize("B,n,levels", [(640, 9000, 0), (700, 60000, 0), (612, 20000, 7), (610, 4096, 0)])
def test_topk_many_rows_one_cta_each(csa2, B, n, levels):
    """Batches of at least 608 rows take one CTA per row (histogram and
    candidates in one pass); ragged n_valid (0, below k, a tile and one more,
    full), planted ties, -inf and NaN must still give the oracle's set."""
    rng = np.random.default_rng(B + n + levels)
    k = 512
    if levels:
        s = rng.integers(0, levels, (B, n)).astype(np.float32)
    else:
        s = rng.standard_normal((B, n)).astype(np.float32)
        s[rng.integers(0, B, 50), rng.integers(0, n, 50)] = 4.25  # ties at the top
    s[0, :64] = -np.inf
    s[1, ::13] = np.nan
    nvalid = rng.integers(1, n + 1, B).astype(np.int32)
    nvalid[:6] = [0, 1, k - 1, 4097 if n > 4097 else n, n, n - 1]
    idx = torch.empty(B, k, dtype=torch.int32, device="cuda")
    csa2.csa2_topk(dev(s), k, idx, csa2.topk_workspace(B, n, k), n_valid=dev(nvalid))
    got = idx.cpu().numpy()
    for b in range(B):
        ref, _ = oracle.topk(s[b, :nvalid[b]], k)
        expect = sorted(int(p) for p in ref if p >= 0)
        assert list(got[b, :len(expect)]) == expect, b
        assert np.all(got[b, len(expect):] == -1), b


def test_topk_one_million_row(csa2):
    rng = np.random.default_rng(9)
    n, k = 1 << 20, 512
    s = rng.standard_normal((1, n)).astype(np.float32)
    s[0, rng.integers(0, n, 40)] = 5.5  # ties at the top
    idx = torch.empty(1, k, dtype=torch.int32, device="cuda")
    csa2.csa2_topk(dev(s), k, idx, csa2.topk_workspace(1, n, k))
    ref, _ = oracle.topk(s[0], k)
    assert list(idx.cpu().numpy()[0]) == sorted(ref.tolist())


def test_topk_with_positions(csa2):
    rng = np.random.default_rng(10)
    B, n, k = 2, 16384, 512
    s = rng.standard_normal((B, n)).astype(np.float32)
    pos = np.stack([rng.permutation(1 << 20)[:n] for _ in range(B)]).astype(np.int32)
    pos[:, ::97] = -1
    idx = torch.empty(B, k, dtype=torch.int32, device="cuda")
    csa2.csa2_topk(dev(s), k, idx, csa2.topk_workspace(B, n, k), positions=dev(pos))
    got = idx.cpu().numpy()
    for b in range(B):
        ref, _ = oracle.topk(s[b], k, positions=pos[b])
        assert list(got[b]) == sorted(ref.tolist())


@pytest.mark.parametrize("n,nbk", [(1 << 17, 2048), (16000, 2048), (1001, 64), (8, 2048)])
def test_block_pool_exact_on_identical_scores(csa2, n, nbk):
    rng = np.random.default_rng(n)
    B = 2
    s = rng.standard_normal((B, n)).astype(np.float32)
    s[1, : n // 3] = 1.0  # ties between block maxima
    nvis = np.array([n, max(1, n - 5)], np.int32)
    pool = torch.empty(B, nbk * 8, dtype=torch.int32, device="cuda")
    csa2.csa2_block_pool(dev(s), dev(nvis), pool, csa2.pool_workspace(B, n, 8, nbk), n_blocks=nbk)
    got = pool.cpu().numpy()
    for b in range(B):
        ref, _ = oracle.block_pool(s[b, :nvis[b]], 8, nbk)
        np.testing.assert_array_equal(got[b], ref)


def test_index_topk_fused_matches_oracle(csa2, case):
    g = case.to_device()
    k = 512
    idx = torch.empty(case.B, k, dtype=torch.int32, device="cuda")
    ws = csa2.index_topk_workspace(case.B, case.cap, k)
    csa2.csa2_index_topk(g["q_data"], g["q_e8m0"], g["w"], g["ik_data"], g["ik_scale"], g["n_visible"], k, idx, ws)
    got = idx.cpu().numpy()
    for b in range(case.B):
        check_topk(case.oracle_scores(b), got[b], k)


def test_index_topk_with_pool_and_reindex(csa2):
    case = DecodeCase(workload=92, Ns=[40000, 17000], reindex=True, planted_blocks=16)
    g = case.to_device()
    k, nbk = 512, 2048
    idx = torch.empty(case.B, k, dtype=torch.int32, device="cuda")
    pool = torch.empty(case.B, nbk * 8, dtype=torch.int32, device="cuda")
    ws = csa2.index_topk_workspace(case.B, case.cap, k, nbk)
    csa2.csa2_index_topk(g["q_data"], g["q_e8m0"], g["w"], g["ik_data"], g["ik_scale"], g["n_visible"], k, idx, ws,
                         pool_blocks=nbk, pool=pool)
    # Reindex layer: its own q scores only the pool
    ridx = torch.empty(case.B, k, dtype=torch.int32, device="cuda")
    rws = csa2.index_topk_workspace(case.B, nbk * 8, k)
    csa2.csa2_index_topk(g["q_re_data"], g["q_re_e8m0"], g["w_re"], g["ik_data"], g["ik_scale"], g["n_visible"], k,
                         ridx, rws, positions=pool)
    got_pool = pool.cpu().numpy()
    got_idx = idx.cpu().numpy()
    got_r = ridx.cpu().numpy()
    for b in range(case.B):
        s = case.oracle_scores(b)
        check_topk(s, got_idx[b], k)
        ref_pool, _ = oracle.block_pool(s, 8, nbk)
        # pool sets agree except blocks whose max is within tolerance of the 2048th block max
        nb = (case.Ns[b] + 7) // 8
        bmax = np.array([s[j * 8:min(case.Ns[b], j * 8 + 8)].max() for j in range(nb)], np.float32)
        gb = set((got_pool[b][got_pool[b] >= 0] // 8).tolist())
        rb = set((ref_pool[ref_pool >= 0] // 8).tolist())
        kth = np.sort(bmax)[::-1][min(nbk, nb) - 1]
        for blk in gb ^ rb:
            assert abs(bmax[blk] - kth) <= 1e-5 * abs(kth)
        # planted blocks are in the pool
        assert set(case.planted[b].tolist()) <= gb
        # Reindex Top-K over the GPU pool against the oracle over the same pool
        pos = got_pool[b]
        rs = oracle.index_score(case.q_re_data[b], case.q_re_e8m0[b], case.w_re[b], case.ik_data[b],
                                case.ik_scale[b], positions=pos)[0]
        check_topk(rs, got_r[b], k, positions=pos)


def test_index_topk_scans_every_tile_once_when_claimed(csa2):
    """Long ragged rows, 8 sequences: past a fixed first range per CTA the
    fused scan's CTAs claim tiles from a per-row counter. The workspace starts
    filled with huge finite scores, so a visible tile that no CTA scored would
    rank first and break the Top-K against the oracle."""
    Ns = [60001, 50000, 65536, 45000, 61234, 58000, 47000, 64000]
    case = DecodeCase(workload=94, Ns=Ns, gen_device="cuda")
    g = case.to_device()
    k = 512
    idx = torch.empty(case.B, k, dtype=torch.int32, device="cuda")
    ws = csa2.index_topk_workspace(case.B, case.cap, k)
    ws.fill_(0x7F)  # every float of the workspace reads 3.39e38
    csa2.csa2_index_topk(g["q_data"], g["q_e8m0"], g["w"], g["ik_data"], g["ik_scale"], g["n_visible"], k, idx, ws)
    torch.cuda.synchronize()
    assert csa2.csa2_get_last_error() == 0
    got = idx.cpu().numpy()
    for b in range(case.B):
        check_topk(case.oracle_scores(b), got[b], k)


def test_claimed_scan_equals_fixed_ranges_and_leaves_counters_zero(csa2):
    """csa2_index_score_claimed gives the bytes csa2_index_score gives (same
    kernel, tiles claimed from counters instead of fixed ranges), on long
    ragged rows where most CTAs claim past a fixed first range, and leaves its
    counters at zero for the next call."""
    Ns = [60001, 50000, 65536, 45000, 61234, 58000, 47000, 64000]
    case = DecodeCase(workload=94, Ns=Ns, gen_device="cuda")
    g = case.to_device()
    ref = torch.empty(case.B, case.cap, dtype=torch.float32, device="cuda")
    csa2.csa2_index_score(g["q_data"], g["q_e8m0"], g["w"], g["ik_data"], g["ik_scale"], g["n_visible"], ref)
    ctr = torch.zeros(2 * case.B, dtype=torch.int32, device="cuda")
    for _ in range(3):
        got = torch.full_like(ref, 3.0e38)
        csa2.csa2_index_score_claimed(g["q_data"], g["q_e8m0"], g["w"], g["ik_data"], g["ik_scale"], g["n_visible"],
                                      got, ctr)
        torch.cuda.synchronize()
        assert csa2.csa2_get_last_error() == 0
        assert torch.equal(got, ref)
        assert int(ctr.abs().sum()) == 0
    # and the scores themselves against the oracle on two rows
    r = ref.cpu().numpy()
    for b in (3, 7):
        s_ = case.oracle_scores(b)
        _scores_close(r[b, :Ns[b]], s_)
        assert np.all(r[b, Ns[b]:] == -np.inf)


def test_claimed_scan_edges(csa2):
    """Claimed scan on a small ragged case: an empty row, a row of one entry,
    rows shorter than the fixed first ranges, n_pos below the capacity; the
    bytes equal the fixed-range scan's and the counters return to zero."""
    case = DecodeCase(workload=95, Ns=[0, 1, 700, 4093, 129])
    g = case.to_device()
    for n_pos in (case.cap, case.cap - 128):
        ref = torch.empty(case.B, n_pos, dtype=torch.float32, device="cuda")
        csa2.csa2_index_score(g["q_data"], g["q_e8m0"], g["w"], g["ik_data"], g["ik_scale"], g["n_visible"], ref)
        ctr = torch.zeros(2 * case.B, dtype=torch.int32, device="cuda")
        got = torch.full_like(ref, 3.0e38)
        csa2.csa2_index_score_claimed(g["q_data"], g["q_e8m0"], g["w"], g["ik_data"], g["ik_scale"], g["n_visible"],
                                      got, ctr)
        torch.cuda.synchronize()
        assert csa2.csa2_get_last_error() == 0
        assert torch.equal(got, ref)
        assert int(ctr.abs().sum()) == 0


def test_prefill_index_score(csa2):
    from fp4_kv_cache_02_gb300.inputs import prefill_chunk
    T, N0 = 6, 2000
    d = prefill_chunk(93, T, N0)
    N = N0 + T
    qd, qs = oracle.quant_mxfp4(d["q_idx"].reshape(-1, 128))
    ikd, iks = oracle.quant_mxfp4(d["ik"])
    scores = torch.empty(T, N, dtype=torch.float32, device="cuda")
    csa2.csa2_prefill_index_score(dev(qd.reshape(T, 32, 64)), dev(qs.reshape(T, 32, 4)), dev(d["w"]), dev(ikd),
                                  dev(iks), N0, scores)
    s = scores.cpu().numpy()
    for t in range(T):
        ref = oracle.index_score(qd.reshape(T, 32, 64)[t], qs.reshape(T, 32, 4)[t], d["w"][t], ikd, iks,
                                 n=N0 + t + 1)[0]
        _scores_close(s[t, :N0 + t + 1], ref)
        assert np.all(s[t, N0 + t + 1:] == -np.inf)


@pytest.mark.parametrize("T,N0", [(37, 9000), (64, 130), (1, 0)])
def test_prefill_index_score_blocks_chunks_and_ragged_edges(csa2, T, N0):
    """Query blocks of 32 with a ragged last block, key chunks of 64 tiles with
    a ragged last tile, and the causal edge running through the tiles."""
    from fp4_kv_cache_02_gb300.inputs import prefill_chunk
    d = prefill_chunk(94, T, N0)
    N = N0 + T
    qd, qs = oracle.quant_mxfp4(d["q_idx"].reshape(-1, 128))
    qd, qs = qd.reshape(T, 32, 64), qs.reshape(T, 32, 4)
    ikd, iks = oracle.quant_mxfp4(d["ik"])
    scores = torch.empty(T, N, dtype=torch.float32, device="cuda")
    csa2.csa2_prefill_index_score(dev(qd), dev(qs), dev(d["w"]), dev(ikd), dev(iks), N0, scores)
    s = scores.cpu().numpy()
    for t in sorted({0, T // 2, T - 1}):
        ref = oracle.index_score(qd[t], qs[t], d["w"][t], ikd, iks, n=N0 + t + 1)[0]
        _scores_close(s[t, :N0 + t + 1], ref)
        assert np.all(s[t, N0 + t + 1:] == -np.inf)


def test_index_score_block_scales_land_on_their_own_rows_and_blocks(csa2):
    """Keys and queries whose 32-channel blocks carry very different power-of-two
    magnitudes: a scale applied to the wrong key row, head or channel block
    changes the score by orders of magnitude."""
    rng = np.random.default_rng(55)
    B, N = 2, 1000
    cap = 1024
    ik = rng.standard_normal((B, N, 128)) * 2.0 ** rng.integers(-12, 12, (B, N, 4)).repeat(32, axis=2)
    q = rng.standard_normal((B, 32, 128)) * 2.0 ** rng.integers(-6, 6, (B, 32, 4)).repeat(32, axis=2)
    from fp4_kv_cache_02_gb300.inputs import bf16_round
    ik, q = bf16_round(ik.astype(np.float32)), bf16_round(q.astype(np.float32))
    w = rng.uniform(0, 1, (B, 32)).astype(np.float32)
    ikd = np.zeros((B, cap, 64), np.uint8)
    iks = np.zeros((B, cap, 4), np.uint8)
    qd = np.zeros((B, 32, 64), np.uint8)
    qs = np.zeros((B, 32, 4), np.uint8)
    for b in range(B):
        ikd[b, :N], iks[b, :N] = oracle.quant_mxfp4(ik[b])
        qd[b], qs[b] = oracle.quant_mxfp4(q[b])
    nv = np.array([N, N - 77], np.int32)
    scores = torch.empty(B, cap, dtype=torch.float32, device="cuda")
    csa2.csa2_index_score(dev(qd), dev(qs), dev(w), dev(ikd), dev(iks), dev(nv), scores)
    s = scores.cpu().numpy()
    for b in range(B):
        ref = oracle.index_score(qd[b], qs[b], w[b], ikd[b], iks[b], n=int(nv[b]))[0]
        _scores_close(s[b, :nv[b]], ref)
        assert np.all(s[b, nv[b]:] == -np.inf)


@pytest.mark.parametrize("mode", ["dense", "pool", "positions"])
def test_index_topk_from_bf16_q_equals_quantise_then_index(csa2, mode):
    """The scan that quantises q itself must give the bytes, scores, indices and
    pool of csa2_quant_mxfp4 followed by csa2_index_topk."""
    case = DecodeCase(workload=88, Ns=[20000, 7000, 130], reindex=(mode == "pool"), planted_blocks=4 if mode == "pool" else 0)
    g = case.to_device()
    B, cap, k = case.B, case.cap, 512
    q16 = g["q_idx"]
    qd = torch.empty(B, 32, 64, dtype=torch.uint8, device="cuda")
    qs = torch.empty(B, 32, 4, dtype=torch.uint8, device="cuda")
    csa2.csa2_quant_mxfp4(q16, qd, qs)
    kw = {}
    n_pos = cap
    if mode == "pool":
        kw = dict(pool_blocks=64)
    if mode == "positions":
        rng = np.random.default_rng(3)
        pos = np.stack([np.sort(rng.choice(cap, 3000, replace=False)) for _ in range(B)]).astype(np.int32)
        pos[:, ::9] = -1
        kw = dict(positions=dev(pos))
        n_pos = 3000
    outs = []
    for fused in (False, True):
        idx = torch.empty(B, k, dtype=torch.int32, device="cuda")
        pool = torch.empty(B, 64 * 8, dtype=torch.int32, device="cuda") if mode == "pool" else None
        ws = csa2.index_topk_workspace(B, n_pos, k, 64 if mode == "pool" else 0)
        ws.fill_(0x5A)
        if fused:
            csa2.csa2_index_topk_bf16(q16, g["w"], g["ik_data"], g["ik_scale"], g["n_visible"], k, idx, ws,
                                      pool=pool, **kw)
        else:
            csa2.csa2_index_topk(qd, qs, g["w"], g["ik_data"], g["ik_scale"], g["n_visible"], k, idx, ws, pool=pool,
                                 **kw)
        torch.cuda.synchronize()
        assert csa2.csa2_get_last_error() == 0
        scores = ws[:B * n_pos * 4].view(torch.float32).view(B, n_pos).clone()
        outs.append((idx.clone(), None if pool is None else pool.clone(), scores))
    assert torch.equal(outs[0][0], outs[1][0])
    if mode == "pool":
        assert torch.equal(outs[0][1], outs[1][1])
    assert torch.equal(outs[0][2], outs[1][2])
