"""The five workloads at full size, in the launch configuration the bench
times, checked against the oracle: every output where the oracle can afford
it, sampled queries where it cannot (the prefill chunk).

  0  decode, 1 sequence, N = 4,096
  1  Full-layer decode, 32 sequences, N = 65,536
  2  Reindex decode with the 2,048 x 8 pool, 8 sequences, N = 1,048,576, planted blocks
  3  prefill chunk, 4,096 queries after 126,976 entries
  4  long-context decode, 4 sequences, N = 1,048,576, 1 Full + 3 Reuse layers
"""

import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_02_gb300.inputs import WORKLOADS, prefill_chunk

from helpers import ATTN_ROW_TOL, DecodeCase, attn_row_error, check_topk, dev

pytestmark = pytest.mark.gpu

K = 512


@pytest.fixture(scope="module")
def csa2():
    from fp4_kv_cache_02_gb300 import csa2 as m
    return m


def _oracle_full_topk(case, b):
    s = case.oracle_scores(b)
    idx, _ = oracle.topk(s, K)
    return s, idx


def _attention_check(csa2, case, g, ref_idx_all, sample):
    B, L = case.B, case.L
    out = torch.empty(B, L, 64, 512, dtype=torch.bfloat16, device="cuda")
    out32 = torch.empty(B, L, 64, 512, dtype=torch.float32, device="cuda")
    ws = csa2.attn_workspace(B * L, K, 128)
    csa2.csa2_sparse_attn_decode(g["Q"], g["kv_data"], g["kv_scale"], g["n_visible"], dev(ref_idx_all), g["swa"],
                                 out, ws, out_f32=out32)
    torch.cuda.synchronize()
    assert csa2.csa2_get_last_error() == 0
    o = out32.cpu().numpy()
    worst = 0.0
    for b in sample:
        for l in range(L):
            ref, _ = case.oracle_attention(b, l, ref_idx_all[b])
            worst = max(worst, attn_row_error(o[b, l], ref))
    assert worst <= ATTN_ROW_TOL, worst
    return worst


@pytest.mark.parametrize("wid", [0, 1, 4])
def test_decode_workload(csa2, wid):
    w = WORKLOADS[wid]
    case = DecodeCase(workload=wid, Ns=[w.N] * w.B, L=w.L, gen_device="cuda" if w.N > 65536 else None)
    g = case.to_device()
    # indexer q quantised on the GPU must equal the oracle's bytes
    qd, qs = csa2.quant_mxfp4(g["q_idx"])
    assert torch.equal(qd.cpu(), torch.from_numpy(case.q_data))
    assert torch.equal(qs.cpu(), torch.from_numpy(case.q_e8m0))
    idx = torch.empty(w.B, K, dtype=torch.int32, device="cuda")
    ws = csa2.index_topk_workspace(w.B, case.cap, K)
    csa2.csa2_index_topk(qd, qs, g["w"], g["ik_data"], g["ik_scale"], g["n_visible"], K, idx, ws)
    got = idx.cpu().numpy()
    ref_idx = np.zeros((w.B, K), np.int32)
    for b in range(w.B):
        s, ref_idx[b] = _oracle_full_topk(case, b)
        check_topk(s, got[b], K, ref_idx=ref_idx[b])
    sample = range(w.B) if w.B <= 4 else [0, 1, w.B // 2, w.B - 1]
    _attention_check(csa2, case, g, ref_idx, sample)


def test_reindex_workload(csa2):
    w = WORKLOADS[2]
    case = DecodeCase(workload=2, Ns=[w.N] * w.B, reindex=True, planted_blocks=w.planted_blocks, gen_device="cuda")
    g = case.to_device()
    nbk = 2048
    idx = torch.empty(w.B, K, dtype=torch.int32, device="cuda")
    pool = torch.empty(w.B, nbk * 8, dtype=torch.int32, device="cuda")
    csa2.csa2_index_topk(g["q_data"], g["q_e8m0"], g["w"], g["ik_data"], g["ik_scale"], g["n_visible"], K, idx,
                         csa2.index_topk_workspace(w.B, case.cap, K, nbk), pool_blocks=nbk, pool=pool)
    ridx = torch.empty(w.B, K, dtype=torch.int32, device="cuda")
    csa2.csa2_index_topk(g["q_re_data"], g["q_re_e8m0"], g["w_re"], g["ik_data"], g["ik_scale"], g["n_visible"], K,
                         ridx, csa2.index_topk_workspace(w.B, nbk * 8, K), positions=pool)
    got_pool, got_idx, got_r = pool.cpu().numpy(), idx.cpu().numpy(), ridx.cpu().numpy()
    ref_r_all = np.zeros((w.B, K), np.int32)
    for b in range(w.B):
        s, ref_idx = _oracle_full_topk(case, b)
        check_topk(s, got_idx[b], K, ref_idx=ref_idx)
        ref_pool, kept = oracle.block_pool(s, 8, nbk)
        assert kept == nbk
        bmax = s.reshape(-1, 8).max(axis=1)
        kth = np.sort(bmax)[::-1][nbk - 1]
        gb = set((got_pool[b] // 8).tolist())
        rb = set((ref_pool // 8).tolist())
        for blk in gb ^ rb:
            assert abs(bmax[blk] - kth) <= 1e-5 * abs(kth)
        assert set(case.planted[b].tolist()) <= gb
        # the Full layer's own Top-512 lies inside its pool
        assert set(got_idx[b].tolist()) <= set(got_pool[b].tolist())
        # Reindex Top-K over the GPU's pool, against the oracle over the same pool
        rs = oracle.index_score(case.q_re_data[b], case.q_re_e8m0[b], case.w_re[b], case.ik_data[b],
                                case.ik_scale[b], positions=got_pool[b])[0]
        ref_r, _ = oracle.topk(rs, K, positions=got_pool[b])
        check_topk(rs, got_r[b], K, positions=got_pool[b], ref_idx=ref_r)
        ref_r_all[b] = ref_r
    _attention_check(csa2, case, g, ref_r_all, [0, 3, 7])


def test_prefill_workload(csa2):
    w = WORKLOADS[3]
    T, N = w.T, w.N
    N0 = N - T
    d = prefill_chunk(3, T, N0, device="cuda")
    qd, qs = oracle.quant_mxfp4(d["q_idx"].reshape(-1, 128))
    qd, qs = qd.reshape(T, 32, 64), qs.reshape(T, 32, 4)
    ikd, iks = oracle.quant_mxfp4(d["ik"])
    kvd, kvs = oracle.pack_kv_fp4(d["kv"])
    swa = oracle.pack_fp8(d["swa"].reshape(-1)).reshape(T + 127, 512)
    gq, gs = csa2.quant_mxfp4(dev(d["q_idx"]).to(torch.bfloat16))
    assert torch.equal(gq.cpu(), torch.from_numpy(qd)) and torch.equal(gs.cpu(), torch.from_numpy(qs))
    scores = torch.empty(T, N, dtype=torch.float32, device="cuda")
    csa2.csa2_prefill_index_score(gq, gs, dev(d["w"]), dev(ikd), dev(iks), N0, scores)
    nvalid = torch.arange(N0 + 1, N0 + T + 1, dtype=torch.int32, device="cuda")
    idx = torch.empty(T, K, dtype=torch.int32, device="cuda")
    csa2.csa2_topk(scores, K, idx, csa2.topk_workspace(T, N, K), n_valid=nvalid)
    got = idx.cpu().numpy()
    del scores
    rng = np.random.default_rng(3)
    sample = sorted(set(list(range(64)) + list(range(T - 64, T)) + rng.choice(T, 128, replace=False).tolist()))
    ref_idx = got.copy()
    for t in sample:
        s = oracle.index_score(qd[t], qs[t], d["w"][t], ikd, iks, n=N0 + t + 1)[0]
        ref_idx[t], _ = oracle.topk(s, K)
        check_topk(s, got[t], K, ref_idx=ref_idx[t])
    out32 = torch.empty(T, 64, 512, dtype=torch.float32, device="cuda")
    out = torch.empty(T, 64, 512, dtype=torch.bfloat16, device="cuda")
    csa2.csa2_sparse_attn_prefill(dev(d["Q"]).to(torch.bfloat16), dev(kvd), dev(kvs), dev(ref_idx), dev(swa), 128,
                                  out, csa2.attn_workspace(T, K, 128), out_f32=out32)
    torch.cuda.synchronize()
    o = out32.cpu().numpy()
    worst = 0.0
    for t in sample[::4]:
        ref, _ = oracle.sparse_attn(d["Q"][t], kvd, kvs, ref_idx[t], swa[t:t + 128])
        worst = max(worst, attn_row_error(o[t], ref))
    assert worst <= ATTN_ROW_TOL, worst
