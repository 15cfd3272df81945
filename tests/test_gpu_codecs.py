"""GPU parity of the FP4/FP8 pack and unpack entry points against the oracle:
bit-exact on random, edge, subnormal, tie and saturating inputs."""

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


def _edge_rows(cols, rng):
    rows = [
        np.zeros(cols), -np.zeros(cols), np.full(cols, 6.0), np.full(cols, 2688.0), np.full(cols, 3000.0),
        np.full(cols, 3.0e38), np.linspace(-5, 5, cols), rng.standard_normal(cols) * 1e-3,
        rng.standard_normal(cols) * 1e4, np.where(np.arange(cols) % 2 == 0, 1e-40, -3.0),
        (2.0 ** rng.integers(-30, 30, cols)) * rng.choice([-1, 1], cols),
        np.tile([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 4.0, -6.0, 0.1, -1e-30, 1e-39, 7.0, 6.5],
                cols // 16),
        np.full(cols, 1e-38), np.full(cols, -2.0 ** -130),
    ]
    return np.stack(rows)


def _inputs(rows, cols, seed):
    rng = np.random.default_rng(seed)
    x = np.concatenate([rng.standard_normal((rows, cols)) * rng.uniform(0.01, 30, (rows, 1)),
                        _edge_rows(cols, rng)])
    return bf16_round(x.astype(np.float32))


@pytest.mark.parametrize("rows", [1, 7, 3000])
def test_quant_mxfp4_bit_exact(csa2, rows):
    x = _inputs(rows, 128, rows)
    ref_d, ref_s = oracle.quant_mxfp4(x)
    xd = dev(x).to(torch.bfloat16)
    data, sc = csa2.quant_mxfp4(xd)
    np.testing.assert_array_equal(data.cpu().numpy(), ref_d)
    np.testing.assert_array_equal(sc.cpu().numpy(), ref_s)
    out = torch.empty(x.shape, dtype=torch.float32, device="cuda")
    csa2.csa2_dequant_mxfp4(data, sc, out)
    np.testing.assert_array_equal(out.cpu().numpy().astype(np.float64), oracle.dequant_mxfp4(ref_d, ref_s))


def test_quant_mxfp4_other_widths(csa2):
    for cols in (32, 96, 512):
        x = _inputs(5, cols, cols)
        ref_d, ref_s = oracle.quant_mxfp4(x)
        data, sc = csa2.quant_mxfp4(dev(x).to(torch.bfloat16))
        np.testing.assert_array_equal(data.cpu().numpy(), ref_d)
        np.testing.assert_array_equal(sc.cpu().numpy(), ref_s)


@pytest.mark.parametrize("n", [1, 13, 4096])
def test_pack_kv_fp4_bit_exact(csa2, n):
    x = _inputs(n, 512, 100 + n)
    ref_d, ref_s = oracle.pack_kv_fp4(x)
    data, sc = csa2.pack_kv_fp4(dev(x).to(torch.bfloat16))
    np.testing.assert_array_equal(data.cpu().numpy(), ref_d)
    np.testing.assert_array_equal(sc.cpu().numpy(), ref_s)
    out = torch.empty(x.shape, dtype=torch.bfloat16, device="cuda")
    csa2.csa2_unpack_kv_fp4(data, sc, out)
    np.testing.assert_array_equal(out.float().cpu().numpy().astype(np.float64), oracle.unpack_kv_fp4(ref_d, ref_s))


@pytest.mark.parametrize("n", [1, 7, 9, 100003])
def test_pack_fp8_bit_exact(csa2, n):
    rng = np.random.default_rng(n)
    x = bf16_round(np.concatenate([rng.standard_normal(n) * 50, [0.0, -0.0, 448.0, 464.0, 500.0, -1e9, 1e-30,
                                                                  2.0 ** -10, -(2.0 ** -9) * 1.5]]).astype(np.float32))
    ref = oracle.pack_fp8(x)
    out = csa2.pack_fp8(dev(x).to(torch.bfloat16))
    np.testing.assert_array_equal(out.cpu().numpy(), ref)
    back = torch.empty(x.shape, dtype=torch.bfloat16, device="cuda")
    csa2.csa2_unpack_fp8_e4m3(out, back)
    np.testing.assert_array_equal(back.float().cpu().numpy().astype(np.float64), oracle.unpack_fp8(ref))


def test_unpack_every_code(csa2):
    codes = np.arange(256, dtype=np.uint8)
    fin = codes[(codes & 0x7F) != 0x7F]
    back = torch.empty(fin.shape, dtype=torch.bfloat16, device="cuda")
    csa2.csa2_unpack_fp8_e4m3(dev(fin), back)
    np.testing.assert_array_equal(back.float().cpu().numpy().astype(np.float64), oracle.unpack_fp8(fin))
    # every (E2M1 byte, E4M3 scale) pair through the main-KV unpacker
    kvd = np.tile(np.arange(256, dtype=np.uint8), 126).reshape(-1, 256)[:, :256]
    kvs = np.repeat(np.arange(126, dtype=np.uint8)[:, None], 32, axis=1)
    kvd = np.ascontiguousarray(kvd[:126])
    out = torch.empty(126, 512, dtype=torch.bfloat16, device="cuda")
    csa2.csa2_unpack_kv_fp4(dev(kvd), dev(kvs), out)
    np.testing.assert_array_equal(out.float().cpu().numpy().astype(np.float64), oracle.unpack_kv_fp4(kvd, kvs))
