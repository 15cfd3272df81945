"""Pins of the oracle's element formats and byte arithmetic against things
other than the oracle itself: torch's E4M3 / E8M0 decoders (library
routines), the pages' printed numbers (tests/golden/page_numbers.json) and
brute-force nearest-value search."""

import json
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))


def g(key):
    return GOLDEN[key]["value"]


def torch_e4m3_values():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def torch_e8m0_values():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()


def test_e4m3_decode_matches_library_for_all_256_codes(orc):
    ref = torch_e4m3_values()
    for c in range(256):
        v = orc.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c] and math.copysign(1, v) == math.copysign(1, ref[c]), c


def test_e8m0_decode_matches_library_for_all_256_codes(orc):
    ref = torch_e8m0_values()
    for c in range(256):
        v = orc.e8m0_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c], c


def test_e2m1_decode_table(orc):
    # The E2M1 grid: zero, the one subnormal 0.5 (half the smallest normal),
    # and the E4M3-representable values (torch decoder) with one mantissa bit
    # from the smallest normal 1 up to the maximum 6 that the report prints
    # (448 x 6 = 2688).
    e4 = torch_e4m3_values()
    normals = sorted({float(v) for v in e4 if not math.isnan(v) and 1.0 <= v <= g("e2m1_max")
                      and (v / 2.0 ** math.floor(math.log2(v))) in (1.0, 1.5)})
    grid = [0.0, normals[0] / 2] + normals
    assert len(grid) == 8 and grid[-1] == 6.0
    vals = [orc.e2m1_value(c) for c in range(16)]
    assert vals[:8] == grid, vals
    assert vals[8:] == [-x for x in grid]
    assert math.copysign(1, vals[8]) < 0  # code 8 is negative zero


def test_max_magnitudes_from_the_report(orc):
    assert orc.e4m3_value(0x7E) == g("e4m3_max")
    assert orc.e2m1_value(7) == g("e2m1_max")
    assert orc.e4m3_value(0x7E) * orc.e2m1_value(7) == g("main_kv_max_magnitude")


def _brute_nearest(x, table):
    """Nearest finite value in `table` (code -> value) to x; ties to the even code."""
    best = None
    for c, v in table.items():
        d = abs(v - x)
        key = (d, c & 1, c)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_e2m1_encode_is_nearest_even_over_a_dense_sweep(orc):
    table = {c: orc.e2m1_value(c) for c in range(8)}
    xs = np.concatenate([np.linspace(0, 7, 2801), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 1e30]])
    for x in xs:
        x = float(np.float32(x))
        expect = _brute_nearest(min(x, 6.0), table)
        assert orc.e2m1_encode(x) == expect, x
        assert orc.e2m1_encode(-x) == (expect | 8), -x


def test_e2m1_tie_cases(orc):
    # ties go to the even code: 0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2.0,
    # 2.5->2.0, 3.5->4.0, 5->4.0
    expect = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for x, c in expect.items():
        assert orc.e2m1_encode(x) == c


def test_e4m3_encode_matches_library_cast_in_range(orc):
    rng = np.random.default_rng(5)
    xs = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(30),
        rng.uniform(-463.9, 463.9, 20000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-2).astype(np.float32),
        np.float32(2.0) ** np.arange(-12, 9, dtype=np.float32),
    ]).astype(np.float32)
    # include every midpoint between neighbouring finite codes (exact ties)
    vals = torch_e4m3_values()[:127]
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    xs = np.concatenate([xs, mids, -mids])
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(x)) for x in xs], np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates(orc):
    for x in (448.0, 463.9, 464.0, 480.0, 1e6, float("inf")):
        assert orc.e4m3_encode(x) == 0x7E
        assert orc.e4m3_encode(-x) == 0xFE
    assert orc.e4m3_encode(float("nan")) == 0x7F
    assert orc.e4m3_encode(-0.0) == 0x80


def test_entry_byte_arithmetic(orc):
    kv = orc.main_kv_entry_bytes()
    ik = orc.indexer_k_entry_bytes()
    assert kv == g("main_kv_entry_bytes")
    assert ik == g("indexer_k_entry_bytes")
    assert kv + ik == g("global_kv_entry_bytes")
    assert kv * 8 / 512 == g("main_kv_bits_per_channel")
    # per token: 3 encoder Full layers at compression m=2, 1 decoder Full at m=1
    per_token = g("full_layers_encoder_m2") * (kv + ik) / 2 + g("full_layers_decoder_m1") * (kv + ik)
    assert per_token == g("global_kv_bytes_per_token")
    # one sequence of 1,048,576 entries of one Full layer
    assert (kv + ik) * (1 << 20) == 373_293_056
