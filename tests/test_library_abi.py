"""CPU checks of the C ABI: the library loads, exports every entry point the
public header declares, and rejects bad arguments on the host (no GPU call)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa2.h")


@pytest.fixture(scope="module")
def lib():
    from fp4_kv_cache_02_gb300 import _build
    path = _build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("csa2_index_score", "csa2_block_pool", "csa2_topk", "csa2_sparse_attn_decode",
                     "csa2_sparse_attn_prefill", "csa2_quant_mxfp4", "csa2_dequant_mxfp4", "csa2_pack_kv_fp4",
                     "csa2_unpack_kv_fp4", "csa2_pack_fp8_e4m3", "csa2_unpack_fp8_e4m3", "csa2_index_topk"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_exposes_the_same_names():
    import fp4_kv_cache_02_gb300.csa2 as b
    for n in declared_functions():
        if n.endswith("_workspace_size") or n in ("csa2_status_string",):
            continue
        assert hasattr(b, n), n


def test_host_argument_checks_without_gpu(lib):
    vp = ctypes.c_void_p
    lib.csa2_quant_mxfp4.argtypes = [vp, ctypes.c_int64, ctypes.c_int32, vp, vp, vp]
    assert lib.csa2_quant_mxfp4(None, 4, 32, None, None, None) == -1
    fake = vp(4096)
    assert lib.csa2_quant_mxfp4(fake, 4, 33, fake, fake, None) == -2
    assert lib.csa2_quant_mxfp4(vp(4097), 4, 32, fake, fake, None) == -3
    assert lib.csa2_quant_mxfp4(fake, 0, 32, fake, fake, None) == 0  # empty: nothing enqueued
    lib.csa2_topk.argtypes = [vp, ctypes.c_int32, ctypes.c_int64, vp, vp, ctypes.c_int32, vp, vp, ctypes.c_size_t, vp]
    assert lib.csa2_topk(fake, 1, 100, None, None, 0, fake, fake, 1 << 20, None) == -2
    assert lib.csa2_topk(fake, 1, 100, None, None, 4097, fake, fake, 1 << 20, None) == -2
    assert lib.csa2_topk(fake, 1, 100, None, None, 8, fake, fake, 16, None) == -6   # workspace too small
    lib.csa2_index_score.argtypes = [vp, vp, vp, ctypes.c_int32, vp, vp, ctypes.c_int64, vp, vp, ctypes.c_int64, vp, vp]
    assert lib.csa2_index_score(fake, fake, fake, 1, fake, fake, 100, fake, None, 100, fake, None) == -3  # cap % 128
    lib.csa2_status_string.restype = ctypes.c_char_p
    assert lib.csa2_status_string(-6) == b"workspace too small or misaligned"


def test_workspace_sizes_are_host_arithmetic(lib):
    lib.csa2_topk_workspace_size.restype = ctypes.c_size_t
    lib.csa2_topk_workspace_size.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int32]
    a = lib.csa2_topk_workspace_size(8, 1 << 20, 512)
    b = lib.csa2_topk_workspace_size(8, 1 << 21, 512)
    assert a > 8 * (1 << 20) * 8 and b > a
    lib.csa2_sparse_attn_workspace_size.restype = ctypes.c_size_t
    lib.csa2_sparse_attn_workspace_size.argtypes = [ctypes.c_int32] * 3
    assert lib.csa2_sparse_attn_workspace_size(32, 512, 128) > 0
