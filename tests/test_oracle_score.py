"""Pins of the oracle's lightning-indexer score
s[j] = sum_h w_h * ReLU(qhat_h . khat_j) against an independent numpy path
(library decoders + float64 matmul), special cases, and the MAC counts the
notes print."""

import json
import os

import numpy as np
import pytest
import torch

from fp4_kv_cache_02_gb300.inputs import bf16_round

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))


def g(key):
    return GOLDEN[key]["value"]


def _decode_mx_independent(orc, data, sc):
    """MXFP4 decode without the oracle's decoder: E2M1 by table, E8M0 by torch."""
    grid = np.array([orc.e2m1_value(c) for c in range(16)])
    lo = data & 0xF
    hi = data >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(*data.shape[:-1], data.shape[-1] * 2)
    e8 = torch.from_numpy(np.ascontiguousarray(sc)).view(torch.float8_e8m0fnu).double().numpy()
    return grid[codes] * np.repeat(e8, 32, axis=-1)


@pytest.fixture(scope="module")
def small_case(orc):
    rng = np.random.default_rng(21)
    n = 300
    q = bf16_round(rng.standard_normal((32, 128)).astype(np.float32))
    w = rng.uniform(0, 1, 32).astype(np.float32)
    k = bf16_round(rng.standard_normal((n, 128)).astype(np.float32))
    qd, qs = orc.quant_mxfp4(q)
    kd, ks = orc.quant_mxfp4(k)
    return dict(q=q, w=w, k=k, qd=qd, qs=qs, kd=kd, ks=ks, n=n)


def test_score_matches_independent_float64_path(orc, small_case):
    c = small_case
    s32, s64, macs = orc.index_score(c["qd"], c["qs"], c["w"], c["kd"], c["ks"])
    qh = _decode_mx_independent(orc, c["qd"], c["qs"])      # [32,128]
    kh = _decode_mx_independent(orc, c["kd"], c["ks"])      # [n,128]
    dots = kh @ qh.T                                        # [n,32], exact in float64
    ref = (np.maximum(dots, 0.0) * c["w"].astype(np.float64)[None, :]).sum(axis=1)
    np.testing.assert_allclose(s64, ref, rtol=1e-14, atol=1e-12)
    assert np.array_equal(s32, s64.astype(np.float32))
    # per-head dots are exact: products of E2M1 values with power-of-two scales
    np.testing.assert_array_equal(dots, np.round(dots * 2.0 ** 40) / 2.0 ** 40)


def test_score_macs_per_pair_is_32_times_128(orc, small_case):
    c = small_case
    _, _, macs = orc.index_score(c["qd"], c["qs"], c["w"], c["kd"], c["ks"])
    assert macs == c["n"] * g("indexer_macs_per_pair")
    assert g("indexer_macs_per_pair") == g("indexer_heads") * g("indexer_head_dim")


def test_model_level_indexer_mac_coefficients(orc, small_case):
    """[B] 4.4: per decoded token the Full layers scan 2.5 'equivalent full
    layers' (3 encoder Full layers over N/2 compressed entries + 1 decoder Full
    layer over N), the 4 Reindex layers scan the 16,384-entry pool."""
    c = small_case
    _, _, macs = orc.index_score(c["qd"], c["qs"], c["w"], c["kd"], c["ks"])
    per_entry = macs // c["n"]
    equivalent_full = g("full_layers_encoder_m2") / 2 + g("full_layers_decoder_m1")
    assert equivalent_full * per_entry == g("indexer_linear_mac_coefficient")
    assert (equivalent_full + g("reindex_layers")) * per_entry == \
        g("indexer_mac_coefficient_without_hierarchy")
    # the linear term at N = 1M is the printed 10.2 G multiply-adds
    assert round(g("indexer_linear_mac_coefficient") * 1e6 / 1e9, 1) == g("indexer_gmac_at_1m")
    assert g("pool_blocks") * g("pool_block_size") == g("pool_positions")


def test_relu_drops_negative_heads(orc):
    k = np.zeros((2, 128), np.float32)
    k[0, :] = 1.0
    k[1, :] = -1.0
    q = np.zeros((32, 128), np.float32)
    q[0, :] = 1.0      # head 0: dot +128 with key 0, -128 with key 1
    q[1, :] = -0.5     # head 1: dot -64 with key 0, +64 with key 1
    w = np.zeros(32, np.float32)
    w[0], w[1] = 0.25, 2.0
    qd, qs = orc.quant_mxfp4(q)
    kd, ks = orc.quant_mxfp4(k)
    s32, s64, _ = orc.index_score(qd, qs, w, kd, ks)
    assert s64[0] == 0.25 * 128
    assert s64[1] == 2.0 * 64


def test_head_weights_pair_with_their_own_head(orc):
    rng = np.random.default_rng(22)
    k = bf16_round(rng.standard_normal((1, 128)).astype(np.float32))
    kd, ks = orc.quant_mxfp4(k)
    kh = _decode_mx_independent(orc, kd, ks)[0]
    q = np.zeros((32, 128), np.float32)
    for h in range(32):
        q[h] = (h + 1) * np.sign(kh) * 0.0625
    qd, qs = orc.quant_mxfp4(q)
    qh = _decode_mx_independent(orc, qd, qs)
    for h in range(32):
        w = np.zeros(32, np.float32)
        w[h] = 1.0
        s32, s64, _ = orc.index_score(qd, qs, w, kd, ks)
        assert s64[0] == max(0.0, float(qh[h] @ kh))


def test_positions_select_rows_and_negative_positions_are_masked(orc, small_case):
    c = small_case
    full32, full64, _ = orc.index_score(c["qd"], c["qs"], c["w"], c["kd"], c["ks"])
    pos = np.array([5, 0, 299, -1, 17], np.int32)
    s32, s64, macs = orc.index_score(c["qd"], c["qs"], c["w"], c["kd"], c["ks"], positions=pos)
    assert np.array_equal(s64[[0, 1, 2, 4]], full64[[5, 0, 299, 17]])
    assert s64[3] == -np.inf
    assert macs == 4 * 4096
