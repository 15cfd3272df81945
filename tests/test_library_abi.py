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
    lib.csa2_index_score_claimed.argtypes = [vp, vp, vp, ctypes.c_int32, vp, vp, ctypes.c_int64, vp, ctypes.c_int64,
                                             vp, vp, vp]
    assert lib.csa2_index_score_claimed(fake, fake, fake, 1, fake, fake, 128, fake, 128, fake, None, None) == -1
    assert lib.csa2_index_score_claimed(fake, fake, fake, 1, fake, fake, 128, fake, 256, fake, fake, None) == -1
    assert lib.csa2_index_score_claimed(fake, fake, fake, 1, fake, fake, 128, fake, 128, fake, vp(4100), None) == -3
    assert lib.csa2_index_score_claimed(fake, fake, fake, 0, fake, fake, 128, fake, 128, fake, fake, None) == 0  # B = 0
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


def test_host_argument_checks_of_the_newer_entry_points(lib):
    """Append, compressor, replay prefill, Bounded-Replay and exchange steps:
    null pointers, bad sizes and misalignment are refused on the host; empty
    work returns OK without enqueuing anything."""
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    fake = vp(1 << 20)
    odd = vp((1 << 20) + 8)
    lib.csa2_kv_append.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, i64, vp, vp, vp]
    assert lib.csa2_kv_append(None, fake, 1, 1, fake, fake, fake, fake, 128, fake, None, None) == -1
    assert lib.csa2_kv_append(fake, fake, -1, 1, fake, fake, fake, fake, 128, fake, None, None) == -1
    assert lib.csa2_kv_append(odd, fake, 1, 1, fake, fake, fake, fake, 128, fake, None, None) == -3
    assert lib.csa2_kv_append(fake, fake, 0, 1, fake, fake, fake, fake, 128, fake, None, None) == 0
    assert lib.csa2_kv_append(fake, fake, 4, 0, fake, fake, fake, fake, 128, fake, fake, None) == 0
    lib.csa2_compress_kv.argtypes = [vp, vp, vp, i64, i32, vp, vp, vp, vp]
    assert lib.csa2_compress_kv(fake, fake, fake, 10, 0, fake, fake, None, None) == -1     # m < 1
    assert lib.csa2_compress_kv(fake, fake, fake, 10, 4, fake, fake, None, None) == -2     # partial block
    assert lib.csa2_compress_kv(odd, fake, fake, 8, 2, fake, fake, None, None) == -3
    assert lib.csa2_compress_kv(fake, fake, fake, 0, 2, fake, fake, None, None) == 0
    lib.csa2_prefill_index_score_compressed.argtypes = [vp, vp, vp, i32, vp, vp, i64, i64, i32, vp, vp]
    # entries visible to the last query beyond the plane: refused
    assert lib.csa2_prefill_index_score_compressed(fake, fake, fake, 8, fake, fake, 100, 200, 2, fake, None) == -1
    assert lib.csa2_prefill_index_score_compressed(fake, fake, fake, 8, fake, fake, 100, 0, 0, fake, None) == -1
    lib.csa2_sparse_attn_prefill_replay.argtypes = [vp, i32, vp, vp, i64, vp, i32, vp, i32, i32, ctypes.c_float,
                                                    vp, vp, vp, vp, sz, vp]
    assert lib.csa2_sparse_attn_prefill_replay(fake, 4, fake, fake, 100, fake, 8, fake, 16, -1, 1.0, fake, None,
                                               None, fake, 1 << 30, None) == -1      # negative replay row
    assert lib.csa2_sparse_attn_prefill_replay(fake, 0, fake, fake, 100, fake, 8, fake, 16, 3, 1.0, fake, None,
                                               None, fake, 1 << 30, None) == 0
    lib.csa2_topk_candidates.argtypes = [vp, i32, i64, vp, vp, i32, i64, vp, vp]
    assert lib.csa2_topk_candidates(fake, 1, 10, None, fake, 0, 0, fake, None) == -1
    assert lib.csa2_topk_candidates(fake, 1, 10, None, fake, 4, 0, vp((1 << 20) + 4), None) == -3
    assert lib.csa2_topk_candidates(fake, 1, 10, None, fake, 4, (1 << 31) - 5, fake, None) == -2
    lib.csa2_topk_merge.argtypes = [vp, i32, i32, i32, i32, vp, vp, sz, vp]
    assert lib.csa2_topk_merge(fake, 2, 1, 8, 0, fake, fake, 1 << 20, None) == -2
    assert lib.csa2_topk_merge(fake, 2, 1, 8, 8, fake, fake, 16, None) == -6
    lib.csa2_shard_positions.argtypes = [vp, i32, i32, i64, i64, vp, vp]
    assert lib.csa2_shard_positions(fake, 1, 8, 10, 5, fake, None) == -1                  # hi < lo
    lib.csa2_shard_pool.argtypes = [vp, i32, i32, i32, i64, i64, vp, vp, vp]
    assert lib.csa2_shard_pool(fake, 1, 8, 0, 0, 8, None, fake, None) == -1
    lib.csa2_attn_merge.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp]
    assert lib.csa2_attn_merge(fake, fake, 0, 1, fake, None, None, None) == -1
    assert lib.csa2_attn_merge(odd, fake, 2, 1, fake, None, None, None) == -3
    assert lib.csa2_attn_merge(fake, fake, 2, 0, fake, None, None, None) == 0
    lib.csa2_block_max.argtypes = [vp, i32, i64, vp, i32, vp, vp]
    assert lib.csa2_block_max(fake, 1, 10, None, 0, fake, None) == -1
    assert lib.csa2_block_max(fake, 0, 10, None, 8, fake, None) == 0
    lib.csa2_index_topk_bf16.argtypes = [vp, vp, i32, vp, vp, i64, vp, vp, i64, i32, vp, i32, vp, vp, sz, vp]
    assert lib.csa2_index_topk_bf16(None, fake, 1, fake, fake, 128, fake, None, 128, 8, fake, 0, None, fake,
                                    1 << 30, None) == -1


def test_merge_workspace_and_launch_counts_are_host_arithmetic(lib):
    lib.csa2_topk_merge_workspace_size.restype = ctypes.c_size_t
    lib.csa2_topk_merge_workspace_size.argtypes = [ctypes.c_int32] * 4
    a = lib.csa2_topk_merge_workspace_size(4, 32, 512, 512)
    assert a >= 2 * 32 * 4 * 512 * 4
    assert lib.csa2_topk_merge_workspace_size(0, 32, 512, 512) == 0
