"""GPU parity of the encoder Full-layer pieces: the softmax-weighted sequence
compressor (bf16 entry within one bf16 rounding of the oracle's fp64 value;
packed bytes bit-exact with the oracle's packing of its own bf16-rounded
entry wherever the fp32 arithmetic cannot flip a bf16 rounding) and the
prefill indexer scan over compressed entries (causal count of complete
entries)."""

import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_02_gb300.inputs import bf16_round, prefill_chunk

from helpers import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    from fp4_kv_cache_02_gb300 import csa2 as m
    return m


@pytest.mark.parametrize("m,n", [(1, 64), (2, 4096), (4, 1000)])
def test_compressor_matches_oracle(csa2, m, n):
    rng = np.random.default_rng(10 * m + 1)
    C = bf16_round((rng.standard_normal((n, 512)) * 2).astype(np.float32))
    Z = bf16_round((rng.standard_normal((n, 512)) * 3).astype(np.float32))
    Z[::5, :64] += 40.0                                  # a dominant token in some blocks
    bias = rng.standard_normal((m, 512)).astype(np.float32)
    n_out = n // m
    kvd = torch.full((n_out + 3, 256), 0xAB, dtype=torch.uint8, device="cuda")
    kvs = torch.full((n_out + 3, 32), 0xAB, dtype=torch.uint8, device="cuda")
    out = torch.empty(n_out, 512, dtype=torch.bfloat16, device="cuda")
    csa2.csa2_compress_kv(dev(C).to(torch.bfloat16), dev(Z).to(torch.bfloat16), dev(bias), m, kvd, kvs, out=out)
    torch.cuda.synchronize()
    assert csa2.csa2_get_last_error() == 0
    got = out.float().cpu().numpy()
    ref = oracle.compress_kv(C, Z, bias, m)
    # fp32 softmax and sum (error a few fp32 ulps of the largest term, up to
    # 2^-20 x max_a |C|, which matters where the terms cancel), then one bf16
    # rounding (at most one bf16 step of the result)
    step = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
    cmax = np.abs(C.astype(np.float64)).reshape(n_out, m, 512).max(axis=1)
    assert np.all(np.abs(got - ref) <= step + 2.0 ** -20 * cmax + 1e-30)
    # end to end: the packed bytes equal the oracle's packing of its own
    # entry rounded to bf16, for every 16-channel block (one E4M3 scale, 8
    # code bytes) whose fp64 values all lie farther than the kernel's fp32
    # error from a bf16 rounding midpoint; a block with a value that close
    # may round either way in fp32 and is checked against the oracle's
    # packing of the kernel's own bf16 entry instead
    gd, gs = kvd[:n_out].cpu().numpy(), kvs[:n_out].cpu().numpy()
    rd, rs = oracle.pack_kv_fp4(oracle.compress_kv_bf16(C, Z, bias, m).astype(np.float32))
    tol = 2.0 ** -20 * cmax + 4 * 2.0 ** -24 * np.abs(ref)
    mid = np.floor(ref / step) * step + step / 2          # the bf16 midpoint inside ref's step
    near = (np.abs(ref - mid) <= tol).reshape(n_out, 32, 16).any(axis=2)   # [entry][block]
    same_d = (gd.reshape(n_out, 32, 8) == rd.reshape(n_out, 32, 8)).all(axis=2)
    same_s = gs == rs
    assert np.all(same_d[~near]) and np.all(same_s[~near])
    print(f"m={m}: {int(near.sum())} of {near.size} blocks within the fp32 error of a bf16 midpoint")
    d, s = oracle.pack_kv_fp4(got)
    kd, ks = d.reshape(n_out, 32, 8), s.reshape(n_out, 32)
    assert np.array_equal(gd.reshape(n_out, 32, 8)[near], kd[near]) and np.array_equal(gs[near], ks[near])
    assert torch.all(kvd[n_out:] == 0xAB) and torch.all(kvs[n_out:] == 0xAB)


def test_compressor_rejects_a_partial_block(csa2):
    x = torch.zeros(5, 512, dtype=torch.bfloat16, device="cuda")
    kvd = torch.zeros(4, 256, dtype=torch.uint8, device="cuda")
    kvs = torch.zeros(4, 32, dtype=torch.uint8, device="cuda")
    with pytest.raises(csa2.Csa2Error):
        csa2.csa2_compress_kv(x, x, torch.zeros(2, 512, device="cuda"), 2, kvd, kvs)


@pytest.mark.parametrize("m,T,p0", [(2, 37, 3001), (2, 64, 0), (4, 33, 517), (1, 5, 700)])
def test_prefill_scan_over_compressed_entries(csa2, m, T, p0):
    d = prefill_chunk(95, T, (p0 + T) // m + 5)          # keys: the compressed entries (synthetic)
    n_entries = (p0 + T) // m + 5
    qd, qs = oracle.quant_mxfp4(d["q_idx"].reshape(-1, 128))
    qd, qs = qd.reshape(T, 32, 64), qs.reshape(T, 32, 4)
    ikd, iks = oracle.quant_mxfp4(d["ik"][:n_entries])
    scores = torch.empty(T, n_entries, dtype=torch.float32, device="cuda")
    csa2.csa2_prefill_index_score_compressed(dev(qd), dev(qs), dev(d["w"]), dev(ikd), dev(iks), p0, m, scores)
    torch.cuda.synchronize()
    assert csa2.csa2_get_last_error() == 0
    s = scores.cpu().numpy()
    for t in sorted({0, 1, T // 2, T - 1}):
        nvis = oracle.compressed_visible(p0 + t, m)
        assert np.all(np.isneginf(s[t, nvis:]))
        if nvis:
            ref = oracle.index_score(qd[t], qs[t], d["w"][t], ikd, iks, n=nvis)[0]
            np.testing.assert_allclose(s[t, :nvis], ref, rtol=1e-5, atol=1e-6 * np.abs(ref).max())
