"""Pins of the oracle's block codecs: MXFP4 (indexer q/K), E2M1 + E4M3-per-16
(main KV) and FP8 E4M3 (SWA), against brute-force nearest-value search,
exact-arithmetic properties and the report's numbers."""

import math

import numpy as np
import pytest
import torch

from fp4_kv_cache_02_gb300.inputs import bf16_round


def _nibbles(row):
    out = []
    for b in row:
        out += [int(b) & 0xF, int(b) >> 4]
    return out


def _brute(x, table):
    best = None
    for c, v in table.items():
        key = (abs(v - x), c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def _edge_rows(rng, cols):
    rows = [
        np.zeros(cols),
        -np.zeros(cols),
        np.full(cols, 6.0),
        np.full(cols, 2688.0),
        np.full(cols, 3000.0),
        np.linspace(-5, 5, cols),
        rng.standard_normal(cols) * 1e-3,
        rng.standard_normal(cols) * 1e4,
        np.where(np.arange(cols) % 2 == 0, 1e-40, -3.0),  # bf16 subnormal next to normal
        (2.0 ** rng.integers(-20, 20, cols)) * rng.choice([-1, 1], cols),
    ]
    return np.stack(rows).astype(np.float32)


@pytest.fixture(scope="module")
def mx_inputs():
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal((40, 128)).astype(np.float32), _edge_rows(rng, 128)])
    return bf16_round(x)


def test_mxfp4_shared_exponent_brackets_amax(orc, mx_inputs):
    data, sc = orc.quant_mxfp4(mx_inputs)
    for r, row in enumerate(mx_inputs):
        for b in range(4):
            blk = row[b * 32:(b + 1) * 32].astype(np.float64)
            amax = np.abs(blk).max()
            X = int(sc[r, b]) - 127
            if amax == 0.0:
                assert X == -127
            elif X > -127:
                # the largest power of two <= amax is 2^(X+2) (E2M1 max exponent is 2)
                assert 2.0 ** (X + 2) <= amax < 2.0 ** (X + 3), (r, b, amax, X)
            else:
                assert amax < 2.0 ** (-127 + 3)


def test_mxfp4_elements_are_nearest_grid_points(orc, mx_inputs):
    data, sc = orc.quant_mxfp4(mx_inputs)
    table = {c: orc.e2m1_value(c) for c in range(8)}
    for r, row in enumerate(mx_inputs):
        codes = _nibbles(data[r])
        for i, x in enumerate(row):
            X = int(sc[r, i // 32]) - 127
            v = math.ldexp(float(x), -X)
            expect = _brute(min(abs(v), 6.0), table) | (8 if math.copysign(1, float(x)) < 0 else 0)
            assert codes[i] == expect, (r, i, x, X)


def test_mxfp4_roundtrip_idempotent(orc, mx_inputs):
    data, sc = orc.quant_mxfp4(mx_inputs)
    deq = orc.dequant_mxfp4(data, sc)
    assert np.all(np.isfinite(deq))
    data2, sc2 = orc.quant_mxfp4(deq.astype(np.float32))
    assert np.array_equal(orc.dequant_mxfp4(data2, sc2), deq)


def test_mxfp4_dequant_uses_library_scale_decoder(orc, mx_inputs):
    data, sc = orc.quant_mxfp4(mx_inputs)
    e8 = torch.from_numpy(sc.copy()).view(torch.float8_e8m0fnu).double().numpy()
    grid = np.array([orc.e2m1_value(c) for c in range(16)])
    codes = np.array([_nibbles(r) for r in data])
    ref = grid[codes] * np.repeat(e8, 32, axis=1)
    assert np.array_equal(orc.dequant_mxfp4(data, sc), ref)


def test_mxfp4_nibble_order_low_first(orc):
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 4.0   # with amax 4: X = 0, element 0 -> code 6 (4.0)
    x[0, 1] = -1.0  # element 1 -> code 0xA (-1.0)
    data, sc = orc.quant_mxfp4(x)
    assert sc[0, 0] == 127
    assert data[0, 0] == 0xA6


@pytest.fixture(scope="module")
def kv_inputs():
    rng = np.random.default_rng(12)
    x = np.concatenate([rng.standard_normal((24, 512)).astype(np.float32),
                        _edge_rows(rng, 512),
                        (rng.standard_normal((4, 512)) * 22.6 / 3).astype(np.float32)])
    return bf16_round(x)


def test_kv_scale_is_nearest_e4m3_to_fp32_amax_over_6(orc, kv_inputs):
    data, sc = orc.pack_kv_fp4(kv_inputs)
    e4 = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    table = {c: float(e4[c]) for c in range(127)}
    for t, row in enumerate(kv_inputs):
        for b in range(32):
            amax = np.float32(np.abs(row[b * 16:(b + 1) * 16]).max())
            q = float(np.float32(amax) / np.float32(6.0))
            expect = _brute(min(q, 448.0), table)
            assert sc[t, b] == expect, (t, b, amax)


def test_kv_elements_are_nearest_grid_points(orc, kv_inputs):
    data, sc = orc.pack_kv_fp4(kv_inputs)
    table = {c: orc.e2m1_value(c) for c in range(8)}
    e4 = torch.from_numpy(sc.copy()).view(torch.float8_e4m3fn).float().numpy()
    for t, row in enumerate(kv_inputs):
        codes = _nibbles(data[t])
        for i, x in enumerate(row):
            s = e4[t, i // 16]
            if s == 0:
                assert codes[i] == 0
                continue
            v = float(np.float32(x) / np.float32(s))
            expect = _brute(min(abs(v), 6.0), table) | (8 if math.copysign(1, float(x)) < 0 else 0)
            assert codes[i] == expect, (t, i, x, s)


def test_kv_dequant_exact_in_bf16_and_bounded_by_2688(orc, kv_inputs):
    data, sc = orc.pack_kv_fp4(kv_inputs)
    deq = orc.unpack_kv_fp4(data, sc)
    # every product of an E2M1 value and an E4M3 scale is exact in bf16
    assert np.array_equal(bf16_round(deq.astype(np.float32)).astype(np.float64), deq)
    assert np.abs(deq).max() <= 2688.0
    # rows filled with 2688 and with 3000 decode to exactly 448 x 6
    assert np.all(deq[24 + 3] == 2688.0)
    assert np.all(deq[24 + 4] == 2688.0)


def test_kv_roundtrip_idempotent(orc, kv_inputs):
    data, sc = orc.pack_kv_fp4(kv_inputs)
    deq = orc.unpack_kv_fp4(data, sc)
    d2, s2 = orc.pack_kv_fp4(deq.astype(np.float32))
    assert np.array_equal(orc.unpack_kv_fp4(d2, s2), deq)


def test_kv_quantisation_error_is_within_half_a_grid_step(orc):
    rng = np.random.default_rng(13)
    x = bf16_round(rng.standard_normal((64, 512)).astype(np.float32))
    data, sc = orc.pack_kv_fp4(x)
    deq = orc.unpack_kv_fp4(data, sc)
    s = np.repeat(torch.from_numpy(sc.copy()).view(torch.float8_e4m3fn).double().numpy(), 16, axis=1)
    # grid spacing is at most 2 (between 4 and 6) times the scale; x/s <= 6 * (1 + 2^-4)
    assert np.all(np.abs(deq - x) <= s * 1.0 + 1e-12 + np.abs(x) * 2.0 ** -4)


def test_fp8_pack_matches_library_cast(orc):
    rng = np.random.default_rng(14)
    x = bf16_round(np.concatenate([rng.standard_normal(50000) * 4, rng.uniform(-460, 460, 5000),
                                   [0.0, -0.0, 1e-30, -1e-30]]).astype(np.float32))
    got = orc.pack_fp8(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)
    assert np.array_equal(orc.unpack_fp8(got),
                          torch.from_numpy(got).view(torch.float8_e4m3fn).double().numpy())


# ---- fused KV append: placement around the pinned codecs ------------------------

def _rows(rng, shape):
    return bf16_round(rng.standard_normal(shape).astype(np.float32) * 3.0)


def test_kv_append_step_by_step_builds_the_bulk_packed_planes(orc):
    """Appending entries a few at a time must give the planes that packing the
    whole sequence at once gives (the bulk codec calls are pinned above)."""
    rng = np.random.default_rng(61)
    B, cap, n = 2, 64, 40
    kv, ik = _rows(rng, (B, n, 512)), _rows(rng, (B, n, 128))
    planes = [np.full((B, cap, w), 0xA5, np.uint8) for w in (256, 32, 64, 4)]
    nv = np.zeros(B, np.int32)
    for lo, hi in ((0, 1), (1, 8), (8, 9), (9, 40)):
        nv = orc.kv_append(kv[:, lo:hi], ik[:, lo:hi], *planes, nv)
        assert list(nv) == [hi, hi]
    for b in range(B):
        d, s = orc.pack_kv_fp4(kv[b])
        qd, qs = orc.quant_mxfp4(ik[b])
        assert np.array_equal(planes[0][b, :n], d) and np.array_equal(planes[1][b, :n], s)
        assert np.array_equal(planes[2][b, :n], qd) and np.array_equal(planes[3][b, :n], qs)
        for pl in planes:
            assert np.all(pl[b, n:] == 0xA5)     # nothing past the visible entries is touched


def test_kv_append_that_does_not_fit_changes_nothing(orc):
    rng = np.random.default_rng(62)
    B, cap, T = 3, 16, 4
    kv, ik = _rows(rng, (B, T, 512)), _rows(rng, (B, T, 128))
    planes = [np.full((B, cap, w), 0x5A, np.uint8) for w in (256, 32, 64, 4)]
    nv = orc.kv_append(kv, ik, *planes, np.array([12, 13, -1], np.int32))
    assert list(nv) == [16, 13, -1]
    assert not np.all(planes[0][0, 12:] == 0x5A)
    for pl in planes:
        assert np.all(pl[1:] == 0x5A)
