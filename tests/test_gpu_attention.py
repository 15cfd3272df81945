"""GPU parity of the sparse attention entry points against the oracle, given
the oracle's index set, plus the closed-form special cases."""

import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_02_gb300.inputs import bf16_round, prefill_chunk

from helpers import ATTN_ROW_TOL, DecodeCase, attn_row_error, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    from fp4_kv_cache_02_gb300 import csa2 as m
    return m


def _run_decode(csa2, g, idx, k, n_swa, B, L):
    out = torch.empty(B, L, 64, 512, dtype=torch.bfloat16, device="cuda")
    out32 = torch.empty(B, L, 64, 512, dtype=torch.float32, device="cuda")
    lse = torch.empty(B, L, 64, dtype=torch.float32, device="cuda")
    ws = csa2.attn_workspace(B * L, k, n_swa)
    csa2.csa2_sparse_attn_decode(g["Q"], g["kv_data"], g["kv_scale"], g["n_visible"], idx,
                                 g["swa"] if n_swa else None, out, ws, out_f32=out32, lse=lse)
    torch.cuda.synchronize()
    assert csa2.csa2_get_last_error() == 0
    return out, out32, lse


def test_decode_attention_matches_oracle(csa2):
    case = DecodeCase(workload=94, Ns=[3000, 700], L=2)
    g = case.to_device()
    k = 512
    rng = np.random.default_rng(1)
    idx = np.stack([rng.permutation(n)[:k] if n >= k else np.concatenate([rng.permutation(n), -np.ones(k - n)])
                    for n in case.Ns]).astype(np.int32)
    idx[0, 10:20] = -1
    out, out32, lse = _run_decode(csa2, g, dev(idx), k, 128, case.B, case.L)
    o32 = out32.cpu().numpy()
    assert torch.equal(out, out32.to(torch.bfloat16))  # bf16 output is the RNE of the fp32 one
    for b in range(case.B):
        for l in range(case.L):
            ref, ref_lse = case.oracle_attention(b, l, idx[b])
            assert attn_row_error(o32[b, l], ref) <= ATTN_ROW_TOL
            np.testing.assert_allclose(lse.cpu().numpy()[b, l], ref_lse, rtol=1e-5, atol=1e-5)
            assert attn_row_error(out.float().cpu().numpy()[b, l], ref) <= ATTN_ROW_TOL + 2.0 ** -8


def _run_reuse(csa2, g, idx, k, n_swa, B, L):
    out = torch.empty(B, L, 64, 512, dtype=torch.bfloat16, device="cuda")
    out32 = torch.empty(B, L, 64, 512, dtype=torch.float32, device="cuda")
    lse = torch.empty(B, L, 64, dtype=torch.float32, device="cuda")
    ws = csa2.attn_workspace(B * L, k, n_swa)
    csa2.csa2_sparse_attn_reuse(g["Q"], g["kv_data"], g["kv_scale"], g["n_visible"], idx,
                                g["swa"] if n_swa else None, out, ws, out_f32=out32, lse=lse)
    torch.cuda.synchronize()
    assert csa2.csa2_get_last_error() == 0
    return out, out32, lse


@pytest.mark.parametrize("L,k,n_swa", [(3, 1024, 128), (4, 512, 128), (4, 512, 40), (2, 300, 256)])
def test_reuse_attention_matches_oracle_and_per_layer_call(csa2, L, k, n_swa):
    """The fused Reuse-layer call (each selected tile gathered once per pair of
    layers) against the oracle, and bit for bit against the per-layer call:
    same partials, same merge order. k = 1024 at L = 3 gives CTAs with two
    items and merge slices that cross a layer boundary; n_swa = 40 a partial
    SWA tile; k = 300 a ragged selected tile with two SWA tiles per layer."""
    case = DecodeCase(workload=93, Ns=[5000, 1500], L=L, n_swa=n_swa)
    g = case.to_device()
    rng = np.random.default_rng(3)
    idx = np.stack([rng.permutation(n)[:k] for n in case.Ns]).astype(np.int32)
    idx[1, 7:31] = -1
    out, out32, lse = _run_reuse(csa2, g, dev(idx), k, n_swa, case.B, case.L)
    o32, l32 = out32.cpu().numpy(), lse.cpu().numpy()
    assert torch.equal(out, out32.to(torch.bfloat16))
    for b in range(case.B):
        for l in range(case.L):
            ref, ref_lse = case.oracle_attention(b, l, idx[b])
            assert attn_row_error(o32[b, l], ref) <= ATTN_ROW_TOL
            np.testing.assert_allclose(l32[b, l], ref_lse, rtol=1e-5, atol=1e-5)
    pout, pout32, plse = _run_decode(csa2, g, dev(idx), k, n_swa, case.B, case.L)
    assert torch.equal(out32, pout32) and torch.equal(lse, plse) and torch.equal(out, pout)


def test_reuse_attention_limits(csa2):
    """L = 1 is the per-layer call; a cluster of 8 CTAs cannot merge 9 layers."""
    case = DecodeCase(workload=92, Ns=[700], L=1)
    g = case.to_device()
    idx = dev(np.arange(64, dtype=np.int32)[None, :] * 5)
    out, out32, lse = _run_reuse(csa2, g, idx, 64, 128, 1, 1)
    pout, pout32, plse = _run_decode(csa2, g, idx, 64, 128, 1, 1)
    assert torch.equal(out32, pout32) and torch.equal(lse, plse)
    q9 = torch.zeros(1, 9, 64, 512, dtype=torch.bfloat16, device="cuda")
    swa9 = torch.zeros(1, 9, 128, 512, dtype=torch.uint8, device="cuda")
    out9 = torch.empty(1, 9, 64, 512, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_sparse_attn_reuse(q9, g["kv_data"], g["kv_scale"], g["n_visible"], idx, swa9, out9,
                                    csa2.attn_workspace(9, 64, 128))
    assert e.value.status == -2


def test_many_queries_walk_their_tiles_on_one_cta(csa2):
    """A launch of many query-layers (here 160 x 1, above four waves of
    5-CTA clusters) runs one CTA per query with an online softmax in tensor
    memory: sampled queries against the oracle, including sequences with
    fewer visible entries than k (-1 entries) and one whose rows are all
    skipped (only its SWA rows remain); then, with no SWA rows, a query with
    no rows at all gives 0 and lse -inf."""
    B = 160
    Ns = [700 + 37 * (b % 9) for b in range(B)]
    case = DecodeCase(workload=91, Ns=Ns, L=1)
    g = case.to_device()
    rng = np.random.default_rng(4)
    k = 512
    idx = np.stack([rng.permutation(n)[:k] for n in Ns]).astype(np.int32)
    idx[5, 100:400] = -1
    idx[17, :] = -1
    out, out32, lse = _run_decode(csa2, g, dev(idx), k, 128, B, 1)
    o32, l32 = out32.cpu().numpy(), lse.cpu().numpy()
    assert torch.equal(out, out32.to(torch.bfloat16))
    for b in (0, 5, 17, 63, 100, 159):
        ref, ref_lse = case.oracle_attention(b, 0, idx[b])
        assert attn_row_error(o32[b, 0], ref) <= ATTN_ROW_TOL
        np.testing.assert_allclose(l32[b, 0], ref_lse, rtol=1e-5, atol=1e-5)
    again, _, _ = _run_decode(csa2, g, dev(idx), k, 128, B, 1)
    assert torch.equal(out, again)
    out0, out0_32, lse0 = _run_decode(csa2, g, dev(idx), k, 0, B, 1)
    assert torch.all(out0_32[17] == 0) and torch.all(lse0[17] == -float("inf"))
    assert np.isfinite(lse0.cpu().numpy()[3]).all()


def test_sequential_mode_rescales_when_a_head_max_jumps(csa2):
    """In the one-CTA-per-query mode a head's P is taken against a reference
    max that moves only when a tile's max passes it by more than 2^8; then O
    is rescaled. Query 3 gets, for head 0, a whole selected tile of rows
    scoring ~14.9 (log2; the other tiles stay near 3) and one later row
    scoring ~24.9, so the reference moves twice, the second time with the
    first tile still weighing ~11 % of the result. Sampled queries against
    the oracle."""
    B = 160
    Ns = [700 + 37 * (b % 9) for b in range(B)]
    case = DecodeCase(workload=91, Ns=Ns, L=1)
    rng = np.random.default_rng(6)
    k = 512
    idx = np.stack([rng.permutation(n)[:k] for n in Ns]).astype(np.int32)
    b = 3
    sgn = np.where(case.Q[b, 0, 0] >= 0, 1.0, -1.0).astype(np.float32)
    for rows, c in ((idx[b, 128:256], 6 * 0.09375), (idx[b, 400:401], 6 * 0.15625)):
        d, sc = oracle.pack_kv_fp4(np.tile(c * sgn, (len(rows), 1)))
        case.kv_data[b, rows], case.kv_scale[b, rows] = d, sc
    g = case.to_device()
    out, out32, lse = _run_decode(csa2, g, dev(idx), k, 128, B, 1)
    o32, l32 = out32.cpu().numpy(), lse.cpu().numpy()
    ref, ref_lse = case.oracle_attention(b, 0, idx[b])
    assert ref_lse[0] * np.log2(np.e) > 20.0      # head 0 is dominated by the planted rows
    for q in (b, 0, 159):
        ref, ref_lse = case.oracle_attention(q, 0, idx[q])
        assert attn_row_error(o32[q, 0], ref) <= ATTN_ROW_TOL
        np.testing.assert_allclose(l32[q, 0], ref_lse, rtol=1e-5, atol=1e-5)


def test_decode_attention_special_cases(csa2):
    case = DecodeCase(workload=95, Ns=[300], n_swa=0)
    g = case.to_device()
    # one selected entry, no SWA rows: the output is that latent, exactly
    idx = np.full((1, 8), -1, np.int32)
    idx[0, 3] = 123
    out, out32, lse = _run_decode(csa2, g, dev(idx), 8, 0, 1, 1)
    row = oracle.unpack_kv_fp4(case.kv_data[0, 123:124], case.kv_scale[0, 123:124])[0]
    np.testing.assert_array_equal(out32.cpu().numpy()[0, 0], np.tile(row, (64, 1)).astype(np.float32))
    # no rows at all: zero output and -inf lse
    idx[0, 3] = -1
    out, out32, lse = _run_decode(csa2, g, dev(idx), 8, 0, 1, 1)
    assert torch.all(out32 == 0) and torch.all(lse == -float("inf"))
    # zero query: the mean of the rows
    g["Q"].zero_()
    idx = np.arange(64, dtype=np.int32)[None, :] * 3
    out, out32, lse = _run_decode(csa2, g, dev(idx), 64, 0, 1, 1)
    rows = oracle.unpack_kv_fp4(case.kv_data[0, idx[0]], case.kv_scale[0, idx[0]])
    np.testing.assert_allclose(out32.cpu().numpy()[0, 0], np.tile(rows.mean(0), (64, 1)), rtol=1e-5, atol=1e-5)


def test_decode_attention_rejects_out_of_range_index(csa2):
    case = DecodeCase(workload=96, Ns=[200])
    g = case.to_device()
    idx = np.arange(8, dtype=np.int32)[None, :]
    idx[0, 2] = 250   # >= n_visible: a device error, the row is skipped
    _ = csa2.csa2_get_last_error()
    out = torch.empty(1, 1, 64, 512, dtype=torch.bfloat16, device="cuda")
    csa2.csa2_sparse_attn_decode(g["Q"], g["kv_data"], g["kv_scale"], g["n_visible"], dev(idx), g["swa"], out,
                                 csa2.attn_workspace(1, 8, 128))
    assert csa2.csa2_get_last_error() == -7
    assert csa2.csa2_get_last_error() == 0  # the error word is cleared


def test_decode_attention_is_deterministic(csa2):
    case = DecodeCase(workload=97, Ns=[2000, 2000])
    g = case.to_device()
    rng = np.random.default_rng(2)
    idx = dev(np.stack([rng.permutation(2000)[:512] for _ in range(2)]).astype(np.int32))
    a, _, _ = _run_decode(csa2, g, idx, 512, 128, 2, 1)
    b, _, _ = _run_decode(csa2, g, idx, 512, 128, 2, 1)
    assert torch.equal(a, b)


@pytest.mark.parametrize("replay_row", [0, 5, 60, 140])
def test_prefill_attention_with_bounded_replay_matches_oracle(csa2, replay_row):
    """Query t at position i = N0 + t sees SWA positions [max(s, i - W + 1), i]
    when the SWA state was replayed from s; swa row r holds position
    N0 - (W - 1) + r, so the replay start maps to row replay_row."""
    T, N0, k, W = 20, 1000, 64, 128
    d = prefill_chunk(97, T, N0)
    kvd, kvs = oracle.pack_kv_fp4(d["kv"])
    swa = oracle.pack_fp8(d["swa"].reshape(-1)).reshape(T + W - 1, 512)
    rng = np.random.default_rng(5)
    idx = np.stack([rng.permutation(N0 + t + 1)[:k] for t in range(T)]).astype(np.int32)
    idx[3, :] = -1                   # a query with SWA rows only (or, when cut away, no rows at all)
    out = torch.empty(T, 64, 512, dtype=torch.bfloat16, device="cuda")
    out32 = torch.empty(T, 64, 512, dtype=torch.float32, device="cuda")
    lse = torch.empty(T, 64, dtype=torch.float32, device="cuda")
    csa2.csa2_sparse_attn_prefill_replay(dev(d["Q"]).to(torch.bfloat16), dev(kvd), dev(kvs), dev(idx), dev(swa), W,
                                         replay_row, out, csa2.attn_workspace(T, k, W), out_f32=out32, lse=lse)
    torch.cuda.synchronize()
    assert csa2.csa2_get_last_error() == 0
    o, l = out32.cpu().numpy(), lse.cpu().numpy()
    s_pos = N0 - (W - 1) + replay_row
    for t in range(T):
        lo, hi = oracle.bounded_replay_window(N0 + t, s_pos, W)
        rows = swa[lo - (N0 - (W - 1)):hi - (N0 - (W - 1))]
        ref, ref_lse = oracle.sparse_attn(d["Q"][t], kvd, kvs, idx[t], rows if len(rows) else None)
        if np.all(np.isneginf(ref_lse)):
            assert np.all(o[t] == 0) and np.all(np.isneginf(l[t]))
            continue
        assert attn_row_error(o[t], ref) <= ATTN_ROW_TOL
        np.testing.assert_allclose(l[t], ref_lse, rtol=1e-5, atol=1e-5)


def test_prefill_attention_matches_oracle(csa2):
    T, N0, k, W = 5, 1000, 64, 128
    d = prefill_chunk(98, T, N0)
    N = N0 + T
    kvd, kvs = oracle.pack_kv_fp4(d["kv"])
    swa = oracle.pack_fp8(d["swa"].reshape(-1)).reshape(T + W - 1, 512)
    rng = np.random.default_rng(4)
    idx = np.stack([rng.permutation(N0 + t + 1)[:k] for t in range(T)]).astype(np.int32)
    out = torch.empty(T, 64, 512, dtype=torch.bfloat16, device="cuda")
    out32 = torch.empty(T, 64, 512, dtype=torch.float32, device="cuda")
    lse = torch.empty(T, 64, dtype=torch.float32, device="cuda")
    csa2.csa2_sparse_attn_prefill(dev(d["Q"]).to(torch.bfloat16), dev(kvd), dev(kvs), dev(idx), dev(swa), W, out,
                                  csa2.attn_workspace(T, k, W), out_f32=out32, lse=lse)
    torch.cuda.synchronize()
    o = out32.cpu().numpy()
    for t in range(T):
        ref, ref_lse = oracle.sparse_attn(d["Q"][t], kvd, kvs, idx[t], swa[t:t + W])
        assert attn_row_error(o[t], ref) <= ATTN_ROW_TOL
        np.testing.assert_allclose(lse.cpu().numpy()[t], ref_lse, rtol=1e-5, atol=1e-5)
