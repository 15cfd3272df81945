"""Pins of the oracle's sparse attention (one softmax over the selected main-KV
latents plus the SWA rows, the latent shared as K and V): closed-form special
cases and an independent float64 numpy softmax on small inputs."""

import numpy as np
import pytest
import torch

from fp4_kv_cache_02_gb300.inputs import bf16_round


def _kv(orc, rng, n):
    x = bf16_round(rng.standard_normal((n, 512)).astype(np.float32))
    return orc.pack_kv_fp4(x)


def _np_attention(q, rows, scale):
    s = scale * (q.astype(np.float64) @ rows.T)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    return (p @ rows) / l, (m + np.log(l))[:, 0]


def _dec_kv_independent(orc, data, sc):
    grid = np.array([orc.e2m1_value(c) for c in range(16)])
    codes = np.stack([data & 0xF, data >> 4], -1).reshape(data.shape[0], 512)
    e4 = torch.from_numpy(np.ascontiguousarray(sc)).view(torch.float8_e4m3fn).double().numpy()
    return grid[codes] * np.repeat(e4, 16, axis=1)


def test_single_entry_no_swa_returns_the_entry(orc):
    rng = np.random.default_rng(41)
    kd, ks = _kv(orc, rng, 10)
    q = bf16_round(rng.standard_normal((4, 512)).astype(np.float32))
    idx = np.array([-1, 7, -1], np.int32)
    out, lse = orc.sparse_attn(q, kd, ks, idx, None)
    row = _dec_kv_independent(orc, kd[7:8], ks[7:8])[0]
    assert np.array_equal(out, np.tile(row, (4, 1)))
    np.testing.assert_allclose(lse, q.astype(np.float64) @ row, rtol=1e-15)


def test_identical_rows_return_that_row(orc):
    rng = np.random.default_rng(42)
    kd, ks = _kv(orc, rng, 1)
    kd = np.repeat(kd, 6, axis=0)
    ks = np.repeat(ks, 6, axis=0)
    q = bf16_round(rng.standard_normal((3, 512)).astype(np.float32))
    out, lse = orc.sparse_attn(q, kd, ks, np.arange(6, dtype=np.int32), None)
    row = _dec_kv_independent(orc, kd[:1], ks[:1])[0]
    np.testing.assert_allclose(out, np.tile(row, (3, 1)), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(lse, q.astype(np.float64) @ row + np.log(6), rtol=1e-13)


def test_zero_query_gives_the_mean_of_selected_and_swa_rows(orc):
    rng = np.random.default_rng(43)
    kd, ks = _kv(orc, rng, 20)
    swa = orc.pack_fp8(bf16_round(rng.standard_normal((5, 512)).astype(np.float32)))
    idx = np.array([3, 11, 19, -1], np.int32)
    q = np.zeros((2, 512), np.float32)
    out, lse = orc.sparse_attn(q, kd, ks, idx, swa)
    rows = np.concatenate([_dec_kv_independent(orc, kd[[3, 11, 19]], ks[[3, 11, 19]]),
                           torch.from_numpy(swa).view(torch.float8_e4m3fn).double().numpy()])
    np.testing.assert_allclose(out[0], rows.mean(axis=0), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, np.log(8.0), rtol=1e-15)


def test_attention_matches_numpy_softmax(orc):
    rng = np.random.default_rng(44)
    kd, ks = _kv(orc, rng, 300)
    swa = orc.pack_fp8(bf16_round(rng.standard_normal((128, 512)).astype(np.float32)))
    q = bf16_round((rng.standard_normal((64, 512)) / np.sqrt(512)).astype(np.float32))
    idx = rng.permutation(300)[:100].astype(np.int32)
    for scale in (1.0, 0.37):
        out, lse = orc.sparse_attn(q, kd, ks, idx, swa, sm_scale=scale)
        rows = np.concatenate([_dec_kv_independent(orc, kd[idx], ks[idx]),
                               torch.from_numpy(swa).view(torch.float8_e4m3fn).double().numpy()])
        ref, ref_lse = _np_attention(q, rows, scale)
        np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lse, ref_lse, rtol=1e-12)


def test_no_rows_gives_zero_and_minus_inf(orc):
    rng = np.random.default_rng(45)
    kd, ks = _kv(orc, rng, 2)
    q = np.ones((2, 512), np.float32)
    out, lse = orc.sparse_attn(q, kd, ks, np.array([-1, -1], np.int32), None)
    assert np.all(out == 0.0) and np.all(lse == -np.inf)


def test_decode_batch_composes_score_topk_attention(orc):
    rng = np.random.default_rng(46)
    B, cap, L = 2, 256, 2
    nvis = np.array([256, 200], np.int32)
    qd = np.zeros((B, 32, 64), np.uint8)
    qs = np.zeros((B, 32, 4), np.uint8)
    ikd = np.zeros((B, cap, 64), np.uint8)
    iks = np.zeros((B, cap, 4), np.uint8)
    kvd = np.zeros((B, cap, 256), np.uint8)
    kvs = np.zeros((B, cap, 32), np.uint8)
    w = rng.uniform(0, 1, (B, 32)).astype(np.float32)
    for b in range(B):
        qd[b], qs[b] = orc.quant_mxfp4(bf16_round(rng.standard_normal((32, 128)).astype(np.float32)))
        ikd[b], iks[b] = orc.quant_mxfp4(bf16_round(rng.standard_normal((cap, 128)).astype(np.float32)))
        kvd[b], kvs[b] = _kv(orc, rng, cap)
    Q = bf16_round((rng.standard_normal((B, L, 64, 512)) / np.sqrt(512)).astype(np.float32))
    swa = np.stack([[orc.pack_fp8(bf16_round(rng.standard_normal((128, 512)).astype(np.float32)))
                     for _ in range(L)] for _ in range(B)])
    idx, out, macs = orc.decode_batch(nvis, qd, qs, w, ikd, iks, kvd, kvs, Q, swa, k=64, n_threads=2)
    assert macs == int(nvis.sum()) * 4096
    for b in range(B):
        s, _, _ = orc.index_score(qd[b], qs[b], w[b], ikd[b], iks[b], n=int(nvis[b]))
        ref_idx, _ = orc.topk(s, 64)
        assert np.array_equal(idx[b], ref_idx)
        for l in range(L):
            o, _ = orc.sparse_attn(Q[b, l], kvd[b], kvs[b], ref_idx, swa[b, l])
            assert np.array_equal(out[b, l], o)


# ---- Bounded Replay ([B] 6): the cut sliding window ------------------------------

def test_bounded_replay_window_properties(orc):
    W = 128
    for i in range(0, 600, 7):
        for s in range(0, i + 1, 5):
            lo, hi = orc.bounded_replay_window(i, s, W)
            vis = list(range(lo, hi))
            assert vis[-1] == i                     # the query's own position is always visible
            assert all(p >= s for p in vis)         # nothing before the replay start
            assert len(vis) == min(W, i - s + 1)    # W positions unless the replay cut is closer
    # a replay start far enough back leaves the plain sliding window
    assert orc.bounded_replay_window(1000, 0, W) == (1000 - W + 1, 1001)
    # replay starting at the query itself: only its own row
    assert orc.bounded_replay_window(50, 50, W) == (50, 51)
