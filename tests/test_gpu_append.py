"""GPU parity of the fused KV append (main-KV latent -> E2M1 + E4M3/16,
indexer key -> MXFP4, written at each sequence's next positions) against the
oracle: bit-exact bytes, untouched bytes elsewhere, the visible counts, and a
decode loop that builds a whole cache entry by entry."""

import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_02_gb300.inputs import bf16_round

from helpers import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    from fp4_kv_cache_02_gb300 import csa2 as m
    return m


def _rows(rng, shape, scale=3.0):
    x = rng.standard_normal(shape).astype(np.float32) * scale
    flat = x.reshape(-1, shape[-1])
    # encoder edge cases: zero blocks, saturating magnitudes, tiny values
    flat[0::7, :32] = 0.0
    flat[1::11, 16:48] *= 1e4
    flat[2::13, 64:96] *= 1e-30
    return bf16_round(x)


def _planes(B, cap, fill):
    return [np.full((B, cap, w), fill, np.uint8) for w in (256, 32, 64, 4)]


def _append(csa2, kv, ik, planes, nv, mode):
    g = [dev(p) for p in planes]
    nvd = dev(nv)
    out = None if mode == "none" else (nvd if mode == "inplace" else torch.full_like(nvd, -7))
    csa2.csa2_kv_append(dev(kv).to(torch.bfloat16), dev(ik).to(torch.bfloat16), *g, nvd, n_visible_out=out)
    torch.cuda.synchronize()
    status = csa2.csa2_get_last_error()
    return [x.cpu().numpy() for x in g], (None if out is None else out.cpu().numpy()), status


@pytest.mark.parametrize("T", [1, 5, 37])
@pytest.mark.parametrize("mode", ["separate", "inplace", "none"])
def test_append_is_bit_exact_with_the_oracle(csa2, T, mode):
    rng = np.random.default_rng(70 + T)
    B, cap = 4, 256
    kv, ik = _rows(rng, (B, T, 512)), _rows(rng, (B, T, 128))
    nv = np.array([0, 17, cap - T, 100], np.int32)
    got, got_nv, status = _append(csa2, kv, ik, _planes(B, cap, 0xC3), nv, mode)
    ref = _planes(B, cap, 0xC3)
    ref_nv = oracle.kv_append(kv, ik, *ref, nv)
    assert status == 0
    for g, r in zip(got, ref):
        assert np.array_equal(g, r)
    if got_nv is not None:
        assert np.array_equal(got_nv, ref_nv)


@pytest.mark.parametrize("mode", ["separate", "inplace"])
def test_bulk_append_takes_two_entries_a_warp(csa2, mode):
    """16,389 entries (an odd count, above the bulk threshold): warps encode
    two entries each, the last one alone; sequence 2 does not fit."""
    rng = np.random.default_rng(75)
    B, T, cap = 3, 5463, 6000
    kv, ik = _rows(rng, (B, T, 512)), _rows(rng, (B, T, 128))
    nv = np.array([0, 537, 600], np.int32)
    got, got_nv, status = _append(csa2, kv, ik, _planes(B, cap, 0x3C), nv, mode)
    ref = _planes(B, cap, 0x3C)
    ref_nv = oracle.kv_append(kv, ik, *ref, nv)
    assert status == -7                               # sequence 2 is dropped and reported
    assert np.array_equal(got_nv, ref_nv)
    for g, r in zip(got, ref):
        assert np.array_equal(g, r)


def test_append_that_does_not_fit_is_dropped_and_reported(csa2):
    rng = np.random.default_rng(80)
    B, cap, T = 3, 128, 6
    kv, ik = _rows(rng, (B, T, 512)), _rows(rng, (B, T, 128))
    nv = np.array([10, cap - 3, 0], np.int32)        # sequence 1 has room for 3 of the 6
    for mode in ("separate", "inplace"):
        got, got_nv, status = _append(csa2, kv, ik, _planes(B, cap, 0x11), nv, mode)
        ref = _planes(B, cap, 0x11)
        ref_nv = oracle.kv_append(kv, ik, *ref, nv)
        assert status == -7                           # CSA2_ERR_DEVICE
        assert np.array_equal(got_nv, ref_nv) and got_nv[1] == cap - 3
        for g, r in zip(got, ref):
            assert np.array_equal(g, r)
    assert csa2.csa2_get_last_error() == 0          # the error word was cleared by the read


def test_decode_loop_builds_the_bulk_packed_cache(csa2):
    """300 decode steps of one entry per sequence, counts advanced in place,
    equal the cache that packing all 300 rows at once gives."""
    rng = np.random.default_rng(81)
    B, cap, n = 3, 384, 300
    kv, ik = _rows(rng, (B, n, 512)), _rows(rng, (B, n, 128))
    g = [torch.zeros(B, cap, w, dtype=torch.uint8, device="cuda") for w in (256, 32, 64, 4)]
    nvd = torch.zeros(B, dtype=torch.int32, device="cuda")
    kvd, ikd = dev(kv).to(torch.bfloat16), dev(ik).to(torch.bfloat16)
    for t in range(n):
        csa2.csa2_kv_append(kvd[:, t:t + 1].contiguous(), ikd[:, t:t + 1].contiguous(), *g, nvd, n_visible_out=nvd)
    torch.cuda.synchronize()
    assert csa2.csa2_get_last_error() == 0
    assert nvd.tolist() == [n] * B
    for b in range(B):
        d, s = oracle.pack_kv_fp4(kv[b])
        qd, qs = oracle.quant_mxfp4(ik[b])
        for got, want in zip(g, (d, s, qd, qs)):
            assert np.array_equal(got[b, :n].cpu().numpy(), want)
            assert torch.all(got[b, n:] == 0)


def test_append_matches_the_library_pack_kernels(csa2):
    """The fused kernel and the standalone pack kernels share the block
    encoders: same bytes for the same rows."""
    rng = np.random.default_rng(82)
    B, T = 2, 64
    kv, ik = _rows(rng, (B, T, 512)), _rows(rng, (B, T, 128))
    got, _, status = _append(csa2, kv, ik, _planes(B, T, 0), np.zeros(B, np.int32), "none")
    assert status == 0
    d, s = csa2.pack_kv_fp4(dev(kv).to(torch.bfloat16))
    qd, qs = csa2.quant_mxfp4(dev(ik).to(torch.bfloat16))
    for g, w in zip(got, (d, s, qd, qs)):
        assert np.array_equal(g, w.cpu().numpy())
