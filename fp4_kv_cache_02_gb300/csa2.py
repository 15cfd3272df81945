"""ctypes binding of libcsa2.so (the CSA2 C ABI declared in include/csa2.h).

Argument marshalling only: every function checks tensor devices, dtypes and
contiguity, passes ``data_ptr()`` values and the CUDA stream handle, and
raises on a non-zero status. All arithmetic runs in the CUDA library. There
is no CPU fallback: importing this module fails if the library is missing.

The ``csa2_*`` functions take caller-allocated output tensors, like the C
ABI. The short-named helpers below them allocate outputs and workspaces with
torch (device memory plumbing) and call the same entry points.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa2.so")

IDX_HEADS = 32
IDX_DIM = 128
HEADS = 64
HEAD_DIM = 512
TOPK = 512
SWA = 128
POOL_BLOCK = 8
POOL_BLOCKS = 2048
CAP_ALIGN = 128
MAX_TOPK = 4096

STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported shape", -3: "misaligned",
          -4: "CUDA error", -5: "device wait timed out", -6: "workspace", -7: "device rejected input",
          -8: "needs more than the static scratch buffer"}
TOPK_STATIC_SCRATCH_BYTES = 32 << 20


class Csa2Error(RuntimeError):
    def __init__(self, name, rc):
        super().__init__(f"{name} failed with status {rc} ({STATUS.get(rc, 'unknown')})")
        self.status = rc


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"CSA2 CUDA library not built ({LIB_PATH} missing); run "
            "`python -c \"import __graft_entry__ as g; g.build()\"` first")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    sig = {
        "csa2_version": (ctypes.c_int, []),
        "csa2_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "csa2_get_last_error": (ctypes.c_int, [vp, ctypes.POINTER(ctypes.c_int)]),
        "csa2_quant_mxfp4": (ctypes.c_int, [vp, i64, i32, vp, vp, vp]),
        "csa2_dequant_mxfp4": (ctypes.c_int, [vp, vp, i64, i32, vp, vp]),
        "csa2_pack_kv_fp4": (ctypes.c_int, [vp, i64, vp, vp, vp]),
        "csa2_unpack_kv_fp4": (ctypes.c_int, [vp, vp, i64, vp, vp]),
        "csa2_pack_fp8_e4m3": (ctypes.c_int, [vp, i64, vp, vp]),
        "csa2_unpack_fp8_e4m3": (ctypes.c_int, [vp, i64, vp, vp]),
        "csa2_kv_append": (ctypes.c_int, [vp, vp, i32, i32, vp, vp, vp, vp, i64, vp, vp, vp]),
        "csa2_index_score": (ctypes.c_int, [vp, vp, vp, i32, vp, vp, i64, vp, vp, i64, vp, vp]),
        "csa2_index_score_claimed": (ctypes.c_int, [vp, vp, vp, i32, vp, vp, i64, vp, i64, vp, vp, vp]),
        "csa2_topk_workspace_size": (sz, [i32, i64, i32]),
        "csa2_topk": (ctypes.c_int, [vp, i32, i64, vp, vp, i32, vp, vp, sz, vp]),
        "csa2_topk_static": (ctypes.c_int, [vp, i32, i64, vp, vp, i32, vp, vp]),
        "csa2_block_pool_workspace_size": (sz, [i32, i64, i32, i32]),
        "csa2_block_pool": (ctypes.c_int, [vp, i32, i64, vp, i32, i32, vp, vp, sz, vp]),
        "csa2_block_max": (ctypes.c_int, [vp, i32, i64, vp, i32, vp, vp]),
        "csa2_topk_candidates": (ctypes.c_int, [vp, i32, i64, vp, vp, i32, i64, vp, vp]),
        "csa2_topk_merge_workspace_size": (sz, [i32, i32, i32, i32]),
        "csa2_topk_merge": (ctypes.c_int, [vp, i32, i32, i32, i32, vp, vp, sz, vp]),
        "csa2_shard_positions": (ctypes.c_int, [vp, i32, i32, i64, i64, vp, vp]),
        "csa2_shard_pool": (ctypes.c_int, [vp, i32, i32, i32, i64, i64, vp, vp, vp]),
        "csa2_attn_merge": (ctypes.c_int, [vp, vp, i32, i32, vp, vp, vp, vp]),
        "csa2_index_topk_workspace_size": (sz, [i32, i64, i32, i32]),
        "csa2_index_topk": (ctypes.c_int, [vp, vp, vp, i32, vp, vp, i64, vp, vp, i64, i32, vp, i32, vp,
                                           vp, sz, vp]),
        "csa2_index_topk_bf16": (ctypes.c_int, [vp, vp, i32, vp, vp, i64, vp, vp, i64, i32, vp, i32, vp, vp, sz,
                                                vp]),
        "csa2_prefill_index_score": (ctypes.c_int, [vp, vp, vp, i32, vp, vp, i64, i64, vp, vp]),
        "csa2_prefill_index_score_compressed": (ctypes.c_int, [vp, vp, vp, i32, vp, vp, i64, i64, i32, vp, vp]),
        "csa2_compress_kv": (ctypes.c_int, [vp, vp, vp, i64, i32, vp, vp, vp, vp]),
        "csa2_sparse_attn_workspace_size": (sz, [i32, i32, i32]),
        "csa2_sparse_attn_kernel_launches": (ctypes.c_int, [i32, i32, i32]),
        "csa2_sparse_attn_decode": (ctypes.c_int, [vp, i32, i32, vp, vp, i64, vp, vp, i32, vp, i32, f32,
                                                   vp, vp, vp, vp, sz, vp]),
        "csa2_sparse_attn_reuse": (ctypes.c_int, [vp, i32, i32, vp, vp, i64, vp, vp, i32, vp, i32, f32,
                                                  vp, vp, vp, vp, sz, vp]),
        "csa2_sparse_attn_prefill": (ctypes.c_int, [vp, i32, vp, vp, i64, vp, i32, vp, i32, f32, vp, vp,
                                                    vp, vp, sz, vp]),
        "csa2_sparse_attn_prefill_replay": (ctypes.c_int, [vp, i32, vp, vp, i64, vp, i32, vp, i32, i32, f32, vp,
                                                           vp, vp, vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()

EXPORTED = [n for n in dir(_lib) if n.startswith("csa2_")]


def lib():
    return _lib


# ---- marshalling helpers -----------------------------------------------------

def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _req(t, dtype, name, allow_none=False):
    if t is None:
        if allow_none:
            return
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _call(name, *args):
    rc = getattr(_lib, name)(*args)
    if rc != 0:
        raise Csa2Error(name, rc)


def csa2_version() -> int:
    return _lib.csa2_version()


def csa2_get_last_error(stream=None) -> int:
    st = ctypes.c_int(0)
    _call("csa2_get_last_error", _s(stream), ctypes.byref(st))
    return st.value


# ---- codecs ------------------------------------------------------------------

def csa2_quant_mxfp4(x, data, e8m0, stream=None):
    _req(x, torch.bfloat16, "x"); _req(data, torch.uint8, "data"); _req(e8m0, torch.uint8, "e8m0")
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    assert data.numel() == rows * cols // 2 and e8m0.numel() == rows * cols // 32
    _call("csa2_quant_mxfp4", _p(x), rows, cols, _p(data), _p(e8m0), _s(stream))


def csa2_dequant_mxfp4(data, e8m0, out, stream=None):
    _req(data, torch.uint8, "data"); _req(e8m0, torch.uint8, "e8m0"); _req(out, torch.float32, "out")
    cols = out.shape[-1]
    rows = out.numel() // cols
    _call("csa2_dequant_mxfp4", _p(data), _p(e8m0), rows, cols, _p(out), _s(stream))


def csa2_pack_kv_fp4(x, kv_data, kv_scale, stream=None):
    _req(x, torch.bfloat16, "x"); _req(kv_data, torch.uint8, "kv_data"); _req(kv_scale, torch.uint8, "kv_scale")
    n = x.numel() // HEAD_DIM
    assert kv_data.numel() == n * 256 and kv_scale.numel() == n * 32
    _call("csa2_pack_kv_fp4", _p(x), n, _p(kv_data), _p(kv_scale), _s(stream))


def csa2_unpack_kv_fp4(kv_data, kv_scale, out, stream=None):
    _req(kv_data, torch.uint8, "kv_data"); _req(kv_scale, torch.uint8, "kv_scale"); _req(out, torch.bfloat16, "out")
    n = out.numel() // HEAD_DIM
    _call("csa2_unpack_kv_fp4", _p(kv_data), _p(kv_scale), n, _p(out), _s(stream))


def csa2_pack_fp8_e4m3(x, out, stream=None):
    _req(x, torch.bfloat16, "x"); _req(out, torch.uint8, "out")
    assert out.numel() == x.numel()
    _call("csa2_pack_fp8_e4m3", _p(x), x.numel(), _p(out), _s(stream))


def csa2_unpack_fp8_e4m3(inp, out, stream=None):
    _req(inp, torch.uint8, "in"); _req(out, torch.bfloat16, "out")
    _call("csa2_unpack_fp8_e4m3", _p(inp), inp.numel(), _p(out), _s(stream))


def csa2_kv_append(kv, ik, kv_data, kv_scale, ik_data, ik_scale, n_visible, n_visible_out=None, stream=None):
    """kv [B,T,512] bf16 (RoPE'd latents), ik [B,T,128] bf16 -> entries at
    n_visible[b] + t of the planes [B,cap,...]; n_visible_out (may be n_visible)."""
    _req(kv, torch.bfloat16, "kv"); _req(ik, torch.bfloat16, "ik")
    for t, n in ((kv_data, "kv_data"), (kv_scale, "kv_scale"), (ik_data, "ik_data"), (ik_scale, "ik_scale")):
        _req(t, torch.uint8, n)
    _req(n_visible, torch.int32, "n_visible"); _req(n_visible_out, torch.int32, "n_visible_out", allow_none=True)
    B, T = kv.shape[0], kv.shape[1]
    _call("csa2_kv_append", _p(kv), _p(ik), B, T, _p(kv_data), _p(kv_scale), _p(ik_data), _p(ik_scale),
          kv_data.shape[1], _p(n_visible), _p(n_visible_out), _s(stream))


def csa2_compress_kv(c, z, bias, m, kv_data, kv_scale, out=None, stream=None):
    """c, z [n_tokens,512] bf16, bias [m,512] fp32 -> entries [n_tokens/m] packed
    into kv_data [.,256] / kv_scale [.,32]; out [n_tokens/m,512] bf16 (optional)."""
    _req(c, torch.bfloat16, "c"); _req(z, torch.bfloat16, "z"); _req(bias, torch.float32, "bias")
    _req(kv_data, torch.uint8, "kv_data"); _req(kv_scale, torch.uint8, "kv_scale")
    _req(out, torch.bfloat16, "out", allow_none=True)
    n_tokens = c.numel() // 512
    n_out = n_tokens // int(m) if int(m) > 0 else 0
    if (z.numel() != c.numel() or bias.numel() < int(m) * 512 or kv_data.numel() < n_out * 256
            or kv_scale.numel() < n_out * 32 or (out is not None and out.numel() < n_out * 512)):
        raise ValueError("csa2_compress_kv: z must match c, bias holds m x 512, and the outputs hold n_tokens / m entries")
    _call("csa2_compress_kv", _p(c), _p(z), _p(bias), n_tokens, int(m), _p(kv_data), _p(kv_scale), _p(out),
          _s(stream))


# ---- indexer, pool, Top-K -----------------------------------------------------

def csa2_index_score(q_data, q_e8m0, w, ik_data, ik_scale, n_visible, scores, positions=None, stream=None):
    """q_data [B,32,64], q_e8m0 [B,32,4], w [B,32]; ik planes [B,cap,64] / [B,cap,4];
    n_visible [B] int32; positions [B,n_pos] or None; scores [B,n_pos] fp32 (out)."""
    for t, n in ((q_data, "q_data"), (q_e8m0, "q_e8m0"), (ik_data, "ik_data"), (ik_scale, "ik_scale")):
        _req(t, torch.uint8, n)
    _req(w, torch.float32, "w"); _req(n_visible, torch.int32, "n_visible"); _req(scores, torch.float32, "scores")
    _req(positions, torch.int32, "positions", allow_none=True)
    B, cap = ik_data.shape[0], ik_data.shape[1]
    n_pos = scores.shape[1]
    _call("csa2_index_score", _p(q_data), _p(q_e8m0), _p(w), B, _p(ik_data), _p(ik_scale), cap,
          _p(n_visible), _p(positions), n_pos, _p(scores), _s(stream))


def csa2_index_score_claimed(q_data, q_e8m0, w, ik_data, ik_scale, n_visible, scores, tile_counters, stream=None):
    """As csa2_index_score without positions; tile_counters [2*B] int32, zero
    before the first call and left zero by every call."""
    for t, n in ((q_data, "q_data"), (q_e8m0, "q_e8m0"), (ik_data, "ik_data"), (ik_scale, "ik_scale")):
        _req(t, torch.uint8, n)
    _req(w, torch.float32, "w"); _req(n_visible, torch.int32, "n_visible"); _req(scores, torch.float32, "scores")
    _req(tile_counters, torch.int32, "tile_counters")
    B, cap = ik_data.shape[0], ik_data.shape[1]
    n_pos = scores.shape[1]
    if tile_counters.numel() < 2 * B:
        raise ValueError("tile_counters needs 2 * B int32")
    _call("csa2_index_score_claimed", _p(q_data), _p(q_e8m0), _p(w), B, _p(ik_data), _p(ik_scale), cap,
          _p(n_visible), n_pos, _p(scores), _p(tile_counters), _s(stream))


def csa2_topk(scores, k, idx, workspace, n_valid=None, positions=None, stream=None):
    _req(scores, torch.float32, "scores"); _req(idx, torch.int32, "idx"); _req(workspace, torch.uint8, "workspace")
    _req(n_valid, torch.int32, "n_valid", allow_none=True); _req(positions, torch.int32, "positions", allow_none=True)
    B, n = scores.shape
    _call("csa2_topk", _p(scores), B, n, _p(n_valid), _p(positions), k, _p(idx), _p(workspace),
          workspace.numel(), _s(stream))


def csa2_topk_static(scores, k, idx, n_valid=None, positions=None, stream=None):
    """csa2_topk without a workspace: for callers that cannot allocate device
    memory. Its scratch is a fixed 32 MiB buffer inside the library, shared by
    all calls (order calls on one stream; overlapping calls race). The first
    call on a device looks the buffer up; make it before any stream capture."""
    _req(scores, torch.float32, "scores"); _req(idx, torch.int32, "idx")
    _req(n_valid, torch.int32, "n_valid", allow_none=True); _req(positions, torch.int32, "positions", allow_none=True)
    B, n = scores.shape
    _call("csa2_topk_static", _p(scores), B, n, _p(n_valid), _p(positions), k, _p(idx), _s(stream))


def csa2_block_pool(scores, n_visible, pool, workspace, block=POOL_BLOCK, n_blocks=POOL_BLOCKS, stream=None):
    _req(scores, torch.float32, "scores"); _req(pool, torch.int32, "pool"); _req(workspace, torch.uint8, "workspace")
    _req(n_visible, torch.int32, "n_visible", allow_none=True)
    B, n = scores.shape
    _call("csa2_block_pool", _p(scores), B, n, _p(n_visible), block, n_blocks, _p(pool), _p(workspace),
          workspace.numel(), _s(stream))


def csa2_index_topk(q_data, q_e8m0, w, ik_data, ik_scale, n_visible, k, idx, workspace, positions=None,
                    n_pos=None, pool_blocks=0, pool=None, stream=None):
    for t, n in ((q_data, "q_data"), (q_e8m0, "q_e8m0"), (ik_data, "ik_data"), (ik_scale, "ik_scale"),
                 (workspace, "workspace")):
        _req(t, torch.uint8, n)
    _req(w, torch.float32, "w"); _req(n_visible, torch.int32, "n_visible"); _req(idx, torch.int32, "idx")
    _req(positions, torch.int32, "positions", allow_none=True); _req(pool, torch.int32, "pool", allow_none=True)
    B, cap = ik_data.shape[0], ik_data.shape[1]
    if n_pos is None:
        n_pos = positions.shape[1] if positions is not None else cap
    _call("csa2_index_topk", _p(q_data), _p(q_e8m0), _p(w), B, _p(ik_data), _p(ik_scale), cap, _p(n_visible),
          _p(positions), n_pos, k, _p(idx), pool_blocks, _p(pool), _p(workspace), workspace.numel(), _s(stream))


def csa2_index_topk_bf16(q, w, ik_data, ik_scale, n_visible, k, idx, workspace, positions=None, n_pos=None,
                         pool_blocks=0, pool=None, stream=None):
    """csa2_index_topk with q [B,32,128] bf16, quantised inside the scan."""
    _req(q, torch.bfloat16, "q")
    for t, n in ((ik_data, "ik_data"), (ik_scale, "ik_scale"), (workspace, "workspace")):
        _req(t, torch.uint8, n)
    _req(w, torch.float32, "w"); _req(n_visible, torch.int32, "n_visible"); _req(idx, torch.int32, "idx")
    _req(positions, torch.int32, "positions", allow_none=True); _req(pool, torch.int32, "pool", allow_none=True)
    B, cap = ik_data.shape[0], ik_data.shape[1]
    if n_pos is None:
        n_pos = positions.shape[1] if positions is not None else cap
    _call("csa2_index_topk_bf16", _p(q), _p(w), B, _p(ik_data), _p(ik_scale), cap, _p(n_visible), _p(positions),
          n_pos, k, _p(idx), pool_blocks, _p(pool), _p(workspace), workspace.numel(), _s(stream))


def csa2_prefill_index_score(q_data, q_e8m0, w, ik_data, ik_scale, p0, scores, stream=None):
    for t, n in ((q_data, "q_data"), (q_e8m0, "q_e8m0"), (ik_data, "ik_data"), (ik_scale, "ik_scale")):
        _req(t, torch.uint8, n)
    _req(w, torch.float32, "w"); _req(scores, torch.float32, "scores")
    T, n_entries = scores.shape
    _call("csa2_prefill_index_score", _p(q_data), _p(q_e8m0), _p(w), T, _p(ik_data), _p(ik_scale), n_entries,
          p0, _p(scores), _s(stream))


def csa2_block_max(scores, bmax, n_visible=None, block=POOL_BLOCK, stream=None):
    """scores [B,n] fp32 -> bmax [B,ceil(n/block)] fp32."""
    _req(scores, torch.float32, "scores"); _req(bmax, torch.float32, "bmax")
    _req(n_visible, torch.int32, "n_visible", allow_none=True)
    B, n = scores.shape
    _call("csa2_block_max", _p(scores), B, n, _p(n_visible), block, _p(bmax), _s(stream))


# ---- context sharding: exchange steps -------------------------------------------

def csa2_topk_candidates(scores, idx, offset, cand, positions=None, stream=None):
    """scores [B,n] fp32, idx [B,k] int32 columns -> cand [B,k,2] int32 pairs
    (fp32 score bits, global position)."""
    _req(scores, torch.float32, "scores"); _req(idx, torch.int32, "idx"); _req(cand, torch.int32, "cand")
    _req(positions, torch.int32, "positions", allow_none=True)
    B, n = scores.shape
    _call("csa2_topk_candidates", _p(scores), B, n, _p(positions), _p(idx), idx.shape[1], int(offset), _p(cand),
          _s(stream))


def csa2_topk_merge(cand, k_out, idx, workspace, stream=None):
    """cand [R,B,k,2] int32 pairs gathered in rank order -> idx [B,k_out] global positions."""
    _req(cand, torch.int32, "cand"); _req(idx, torch.int32, "idx"); _req(workspace, torch.uint8, "workspace")
    R, B, k = cand.shape[0], cand.shape[1], cand.shape[2]
    _call("csa2_topk_merge", _p(cand), R, B, k, k_out, _p(idx), _p(workspace), workspace.numel(), _s(stream))


def csa2_shard_positions(idx, lo, hi, local_idx, stream=None):
    _req(idx, torch.int32, "idx"); _req(local_idx, torch.int32, "local_idx")
    B, k = idx.shape
    _call("csa2_shard_positions", _p(idx), B, k, int(lo), int(hi), _p(local_idx), _s(stream))


def csa2_shard_pool(blocks, lo, hi, pool, n_visible=None, block=POOL_BLOCK, stream=None):
    _req(blocks, torch.int32, "blocks"); _req(pool, torch.int32, "pool")
    _req(n_visible, torch.int32, "n_visible", allow_none=True)
    B, nb = blocks.shape
    _call("csa2_shard_pool", _p(blocks), B, nb, block, int(lo), int(hi), _p(n_visible), _p(pool), _s(stream))


def csa2_attn_merge(parts, lses, out, out_f32=None, lse_out=None, stream=None):
    """parts [R,...,64,512] fp32, lses [R,...,64] fp32 -> out [...,64,512] bf16."""
    _req(parts, torch.float32, "parts"); _req(lses, torch.float32, "lses"); _req(out, torch.bfloat16, "out")
    _req(out_f32, torch.float32, "out_f32", allow_none=True); _req(lse_out, torch.float32, "lse_out", allow_none=True)
    R = parts.shape[0]
    n_q = parts[0].numel() // (HEADS * HEAD_DIM)
    _call("csa2_attn_merge", _p(parts), _p(lses), R, n_q, _p(out), _p(out_f32), _p(lse_out), _s(stream))


def csa2_prefill_index_score_compressed(q_data, q_e8m0, w, ik_data, ik_scale, p0, m, scores, stream=None):
    for t, n in ((q_data, "q_data"), (q_e8m0, "q_e8m0"), (ik_data, "ik_data"), (ik_scale, "ik_scale")):
        _req(t, torch.uint8, n)
    _req(w, torch.float32, "w"); _req(scores, torch.float32, "scores")
    T, n_entries = scores.shape
    _call("csa2_prefill_index_score_compressed", _p(q_data), _p(q_e8m0), _p(w), T, _p(ik_data), _p(ik_scale),
          n_entries, int(p0), int(m), _p(scores), _s(stream))


# ---- attention ------------------------------------------------------------------

def csa2_sparse_attn_kernel_launches(n_queries, k, n_swa) -> int:
    """Kernel launches one attention call makes on the current device."""
    return int(_lib.csa2_sparse_attn_kernel_launches(n_queries, k, n_swa))


def csa2_sparse_attn_decode(q, kv_data, kv_scale, n_visible, idx, swa, out, workspace, out_f32=None, lse=None,
                            sm_scale=1.0, stream=None):
    """q [B,L,64,512] bf16; kv planes [B,cap,256]/[B,cap,32]; idx [B,k]; swa [B,L,n_swa,512] u8."""
    _req(q, torch.bfloat16, "q"); _req(kv_data, torch.uint8, "kv_data"); _req(kv_scale, torch.uint8, "kv_scale")
    _req(n_visible, torch.int32, "n_visible"); _req(idx, torch.int32, "idx"); _req(out, torch.bfloat16, "out")
    _req(workspace, torch.uint8, "workspace"); _req(swa, torch.uint8, "swa", allow_none=True)
    _req(out_f32, torch.float32, "out_f32", allow_none=True); _req(lse, torch.float32, "lse", allow_none=True)
    B, L = q.shape[0], q.shape[1]
    cap = kv_data.shape[1]
    k = idx.shape[1]
    n_swa = swa.shape[2] if swa is not None else 0
    _call("csa2_sparse_attn_decode", _p(q), B, L, _p(kv_data), _p(kv_scale), cap, _p(n_visible), _p(idx), k,
          _p(swa), n_swa, float(sm_scale), _p(out), _p(out_f32), _p(lse), _p(workspace), workspace.numel(),
          _s(stream))


def csa2_sparse_attn_reuse(q, kv_data, kv_scale, n_visible, idx, swa, out, workspace, out_f32=None, lse=None,
                           sm_scale=1.0, stream=None):
    """As csa2_sparse_attn_decode, with each selected tile gathered once for a
    pair of the L Reuse layers (bit-identical results)."""
    _req(q, torch.bfloat16, "q"); _req(kv_data, torch.uint8, "kv_data"); _req(kv_scale, torch.uint8, "kv_scale")
    _req(n_visible, torch.int32, "n_visible"); _req(idx, torch.int32, "idx"); _req(out, torch.bfloat16, "out")
    _req(workspace, torch.uint8, "workspace"); _req(swa, torch.uint8, "swa", allow_none=True)
    _req(out_f32, torch.float32, "out_f32", allow_none=True); _req(lse, torch.float32, "lse", allow_none=True)
    B, L = q.shape[0], q.shape[1]
    cap = kv_data.shape[1]
    k = idx.shape[1]
    n_swa = swa.shape[2] if swa is not None else 0
    _call("csa2_sparse_attn_reuse", _p(q), B, L, _p(kv_data), _p(kv_scale), cap, _p(n_visible), _p(idx), k,
          _p(swa), n_swa, float(sm_scale), _p(out), _p(out_f32), _p(lse), _p(workspace), workspace.numel(),
          _s(stream))


def csa2_sparse_attn_prefill(q, kv_data, kv_scale, idx, swa, n_swa, out, workspace, out_f32=None, lse=None,
                             sm_scale=1.0, stream=None):
    """q [T,64,512] bf16; kv planes [n_entries,256]/[n_entries,32]; idx [T,k];
    swa [T+n_swa-1,512] u8 (query t uses rows t..t+n_swa-1)."""
    _req(q, torch.bfloat16, "q"); _req(kv_data, torch.uint8, "kv_data"); _req(kv_scale, torch.uint8, "kv_scale")
    _req(idx, torch.int32, "idx"); _req(out, torch.bfloat16, "out"); _req(workspace, torch.uint8, "workspace")
    _req(swa, torch.uint8, "swa", allow_none=True)
    _req(out_f32, torch.float32, "out_f32", allow_none=True); _req(lse, torch.float32, "lse", allow_none=True)
    T = q.shape[0]
    n_entries = kv_data.shape[0]
    k = idx.shape[1]
    _call("csa2_sparse_attn_prefill", _p(q), T, _p(kv_data), _p(kv_scale), n_entries, _p(idx), k, _p(swa), n_swa,
          float(sm_scale), _p(out), _p(out_f32), _p(lse), _p(workspace), workspace.numel(), _s(stream))


def csa2_sparse_attn_prefill_replay(q, kv_data, kv_scale, idx, swa, n_swa, replay_row, out, workspace, out_f32=None,
                                    lse=None, sm_scale=1.0, stream=None):
    """csa2_sparse_attn_prefill with the Bounded-Replay cut: query t uses swa
    rows max(t, replay_row) .. t + n_swa - 1."""
    _req(q, torch.bfloat16, "q"); _req(kv_data, torch.uint8, "kv_data"); _req(kv_scale, torch.uint8, "kv_scale")
    _req(idx, torch.int32, "idx"); _req(out, torch.bfloat16, "out"); _req(workspace, torch.uint8, "workspace")
    _req(swa, torch.uint8, "swa", allow_none=True)
    _req(out_f32, torch.float32, "out_f32", allow_none=True); _req(lse, torch.float32, "lse", allow_none=True)
    T = q.shape[0]
    n_entries = kv_data.shape[0]
    k = idx.shape[1]
    _call("csa2_sparse_attn_prefill_replay", _p(q), T, _p(kv_data), _p(kv_scale), n_entries, _p(idx), k, _p(swa),
          n_swa, int(replay_row), float(sm_scale), _p(out), _p(out_f32), _p(lse), _p(workspace), workspace.numel(),
          _s(stream))


# ---- allocating helpers (torch memory plumbing + the entry points above) --------

def _ws(nbytes, device):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def quant_mxfp4(x, stream=None):
    rows = x.numel() // x.shape[-1]
    data = torch.empty(*x.shape[:-1], x.shape[-1] // 2, dtype=torch.uint8, device=x.device)
    sc = torch.empty(*x.shape[:-1], x.shape[-1] // 32, dtype=torch.uint8, device=x.device)
    csa2_quant_mxfp4(x, data, sc, stream)
    return data, sc


def pack_kv_fp4(x, stream=None):
    data = torch.empty(*x.shape[:-1], 256, dtype=torch.uint8, device=x.device)
    sc = torch.empty(*x.shape[:-1], 32, dtype=torch.uint8, device=x.device)
    csa2_pack_kv_fp4(x, data, sc, stream)
    return data, sc


def pack_fp8(x, stream=None):
    out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    csa2_pack_fp8_e4m3(x, out, stream)
    return out


def topk_workspace(B, n, k, device="cuda"):
    return _ws(_lib.csa2_topk_workspace_size(B, n, k), device)


def pool_workspace(B, n, block=POOL_BLOCK, n_blocks=POOL_BLOCKS, device="cuda"):
    return _ws(_lib.csa2_block_pool_workspace_size(B, n, block, n_blocks), device)


def index_topk_workspace(B, n_pos, k, pool_blocks=0, device="cuda"):
    return _ws(_lib.csa2_index_topk_workspace_size(B, n_pos, k, pool_blocks), device)


def merge_workspace(R, B, k, k_out, device="cuda"):
    return _ws(_lib.csa2_topk_merge_workspace_size(R, B, k, k_out), device)


def attn_workspace(n_queries, k, n_swa, device="cuda"):
    return _ws(_lib.csa2_sparse_attn_workspace_size(n_queries, k, n_swa), device)
