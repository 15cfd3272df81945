"""Pins of the oracle's sequence compressor (every m tokens merge into one
entry by a per-channel softmax over the group of Z + bias weighting C) and of
the causal count of complete compressed entries: closed forms and limits."""

import numpy as np
import pytest

import oracle


def _rand(rng, shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def test_m1_is_the_identity():
    rng = np.random.default_rng(1)
    C, Z, b = _rand(rng, (9, 16)), _rand(rng, (9, 16)), _rand(rng, (1, 16))
    assert np.array_equal(oracle.compress_kv(C, Z, b, 1), C)


@pytest.mark.parametrize("m", [2, 3, 4])
def test_equal_logits_give_the_block_mean(m):
    rng = np.random.default_rng(m)
    n = 6 * m
    C = _rand(rng, (n, 32))
    Z = np.repeat(_rand(rng, (n // m, 32)), m, axis=0)    # equal within each block
    out = oracle.compress_kv(C, Z, np.zeros((m, 32)), m)
    np.testing.assert_allclose(out, C.reshape(n // m, m, 32).mean(axis=1), rtol=1e-13, atol=1e-14)


def test_shift_invariance_within_a_block():
    rng = np.random.default_rng(5)
    m, n = 2, 20
    C, Z, b = _rand(rng, (n, 8)), _rand(rng, (n, 8)), _rand(rng, (m, 8))
    shift = np.repeat(_rand(rng, (n // m, 8), 50.0), m, axis=0)
    np.testing.assert_allclose(oracle.compress_kv(C, Z + shift, b, m), oracle.compress_kv(C, Z, b, m),
                               rtol=1e-12, atol=1e-13)


def test_dominant_token_and_bias_select_that_token():
    rng = np.random.default_rng(6)
    m, n, D = 4, 12, 8
    C, Z = _rand(rng, (n, D)), _rand(rng, (n, D))
    # a bias that strongly favours position 2 of every block, channel by channel
    b = np.zeros((m, D))
    b[2, :] = 1000.0
    out = oracle.compress_kv(C, Z, b, m)
    np.testing.assert_allclose(out, C.reshape(n // m, m, D)[:, 2, :], rtol=1e-12)
    # a logit that favours a different token in each channel
    Z2 = np.zeros((n, D))
    for c in range(D):
        Z2[(c % m)::m, c] = 1000.0
    out2 = oracle.compress_kv(C, Z2, np.zeros((m, D)), m)
    want = np.stack([C.reshape(n // m, m, D)[:, c % m, c] for c in range(D)], axis=1)
    np.testing.assert_allclose(out2, want, rtol=1e-12)


def test_two_token_weights_are_a_logistic():
    rng = np.random.default_rng(7)
    C, Z, b = _rand(rng, (2, 5)), _rand(rng, (2, 5)), _rand(rng, (2, 5))
    d = (Z[0] + b[0]) - (Z[1] + b[1])
    w0 = 1.0 / (1.0 + np.exp(-d))
    np.testing.assert_allclose(oracle.compress_kv(C, Z, b, 2)[0], w0 * C[0] + (1 - w0) * C[1], rtol=1e-12)


def test_compressed_visible_counts_complete_entries():
    assert [oracle.compressed_visible(p, 1) for p in range(5)] == [1, 2, 3, 4, 5]
    assert [oracle.compressed_visible(p, 2) for p in range(6)] == [0, 1, 1, 2, 2, 3]
    assert [oracle.compressed_visible(p, 4) for p in range(9)] == [0, 0, 0, 1, 1, 1, 1, 2, 2]


def test_bf16_rounding_matches_the_library_cast():
    # float32 inputs are exact in float64: the oracle's rounding must equal
    # torch's round-to-nearest-even float32 -> bfloat16 cast, ties included
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(13)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-30, 30, 200000))).astype(np.float32)
    bits = x.view(np.uint32)
    ties = ((bits & ~np.uint32(0xFFFF)) | np.uint32(0x8000)).view(np.float32)   # exactly half a bf16 step
    for v in (x, ties, np.array([0.0, -0.0, 1.0, -1.0, 3.0, 255.0, 257.0, 65280.0], np.float32)):
        ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
        assert np.array_equal(oracle.bf16_rne(v.astype(np.float64)), ref)


def test_bf16_rounding_of_values_between_float32_neighbours():
    # a float64 just above a bf16 midpoint rounds up even where float32 would
    # first round it onto the midpoint (no double rounding)
    mid = 1.0 + 2.0 ** -8                           # halfway between bf16 1 and 1 + 2^-7
    assert oracle.bf16_rne(mid) == 1.0              # tie to even
    assert oracle.bf16_rne(mid + 2.0 ** -40) == 1.0 + 2.0 ** -7
    assert oracle.bf16_rne(mid - 2.0 ** -40) == 1.0
    assert oracle.bf16_rne(-(mid + 2.0 ** -40)) == -(1.0 + 2.0 ** -7)
