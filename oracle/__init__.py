"""CPU oracle for the CSA2 hot path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` leg of
``bench.py`` may import this package. The CUDA library never calls it and
shares no code with it. The arithmetic lives in ``csa2_oracle.c`` (plain C,
double accumulation); this module compiles it with gcc on first use and
exposes numpy-facing wrappers.

Sources cited in the C file:
  [R]  "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression"
       (technical-report digest)
  [B]  "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression"
       (mer.dev reading notes)
  [V4] "DeepSeek-V4: Towards Highly Efficient Million-Token Context
       Intelligence" (paperglide summary)

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, library routines, brute force or the pages' numbers.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa2_oracle.c")
_HDR = os.path.join(_HERE, "csa2_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

IDX_HEADS = 32
IDX_DIM = 128
KV_DIM = 512


def build(force: bool = False) -> str:
    """Compile csa2_oracle.c into liboracle.so (gcc, OpenMP). Returns the path."""
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            d, i64, i32, u8p, f32p, f64p, i32p = (
                ctypes.c_double, ctypes.c_int64, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p)
            L.orc_e2m1_value.restype = d
            L.orc_e2m1_value.argtypes = [ctypes.c_uint]
            L.orc_e4m3_value.restype = d
            L.orc_e4m3_value.argtypes = [ctypes.c_uint]
            L.orc_e8m0_value.restype = d
            L.orc_e8m0_value.argtypes = [ctypes.c_uint]
            L.orc_e2m1_encode.restype = ctypes.c_uint
            L.orc_e2m1_encode.argtypes = [ctypes.c_float]
            L.orc_e4m3_encode.restype = ctypes.c_uint
            L.orc_e4m3_encode.argtypes = [ctypes.c_float]
            L.orc_quant_mxfp4.argtypes = [f32p, i64, i32, u8p, u8p]
            L.orc_dequant_mxfp4.argtypes = [u8p, u8p, i64, i32, f64p]
            L.orc_pack_kv_fp4.argtypes = [f32p, i64, u8p, u8p]
            L.orc_unpack_kv_fp4.argtypes = [u8p, u8p, i64, f64p]
            L.orc_pack_fp8.argtypes = [f32p, i64, u8p]
            L.orc_unpack_fp8.argtypes = [u8p, i64, f64p]
            L.orc_main_kv_entry_bytes.restype = i32
            L.orc_indexer_k_entry_bytes.restype = i32
            L.orc_index_score.restype = ctypes.c_uint64
            L.orc_index_score.argtypes = [u8p, u8p, f32p, u8p, u8p, i32p, i64, f32p, f64p]
            L.orc_topk.restype = i32
            L.orc_topk.argtypes = [f32p, i32p, i64, i32, i32p]
            L.orc_block_pool.restype = i32
            L.orc_block_pool.argtypes = [f32p, i64, i32, i32, i32p]
            L.orc_block_max.argtypes = [f32p, i64, i32, f32p]
            L.orc_compress_kv.argtypes = [f64p, f64p, f64p, i64, i32, i32, f64p]
            L.orc_attn_merge.argtypes = [f64p, f64p, i32, i32, i32, f64p, f64p]
            L.orc_sparse_attn.argtypes = [f32p, i32, i32, u8p, u8p, i32p, i32, u8p, i32, d, f64p, f64p]
            L.orc_decode_batch.restype = ctypes.c_uint64
            L.orc_decode_batch.argtypes = [i32, i64, i32p, u8p, u8p, f32p, u8p, u8p, u8p, u8p,
                                           i32, i32, f32p, i32, i32, u8p, i32, d, i32p, f64p, i32]
            L.orc_max_threads.restype = i32
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- element formats --------------------------------------------------------

def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(code)


def e8m0_value(code: int) -> float:
    return lib().orc_e8m0_value(code)


def e2m1_encode(x: float) -> int:
    return lib().orc_e2m1_encode(x)


def e4m3_encode(x: float) -> int:
    return lib().orc_e4m3_encode(x)


# ---- codecs -----------------------------------------------------------------

def quant_mxfp4(x):
    """x: float32 [rows, cols] (cols % 32 == 0) -> (data u8 [rows, cols/2], e8m0 u8 [rows, cols/32])."""
    x = _c(x, np.float32)
    rows, cols = x.shape
    assert cols % 32 == 0
    data = np.zeros((rows, cols // 2), np.uint8)
    sc = np.zeros((rows, cols // 32), np.uint8)
    lib().orc_quant_mxfp4(_p(x), rows, cols, _p(data), _p(sc))
    return data, sc


def dequant_mxfp4(data, e8m0):
    data = _c(data, np.uint8)
    e8m0 = _c(e8m0, np.uint8)
    rows = data.shape[0]
    cols = data.shape[1] * 2
    out = np.zeros((rows, cols), np.float64)
    lib().orc_dequant_mxfp4(_p(data), _p(e8m0), rows, cols, _p(out))
    return out


def pack_kv_fp4(x):
    """x: float32 [n, 512] -> (kv_data u8 [n, 256], kv_scale u8 [n, 32])."""
    x = _c(x, np.float32)
    n = x.shape[0]
    assert x.shape[1] == KV_DIM
    data = np.zeros((n, KV_DIM // 2), np.uint8)
    sc = np.zeros((n, KV_DIM // 16), np.uint8)
    lib().orc_pack_kv_fp4(_p(x), n, _p(data), _p(sc))
    return data, sc


def unpack_kv_fp4(kv_data, kv_scale):
    kv_data = _c(kv_data, np.uint8)
    kv_scale = _c(kv_scale, np.uint8)
    n = kv_data.shape[0]
    out = np.zeros((n, KV_DIM), np.float64)
    lib().orc_unpack_kv_fp4(_p(kv_data), _p(kv_scale), n, _p(out))
    return out


def pack_fp8(x):
    x = _c(x, np.float32)
    out = np.zeros(x.shape, np.uint8)
    lib().orc_pack_fp8(_p(x), x.size, _p(out))
    return out


def unpack_fp8(b):
    b = _c(b, np.uint8)
    out = np.zeros(b.shape, np.float64)
    lib().orc_unpack_fp8(_p(b), b.size, _p(out))
    return out


def kv_append(kv, ik, kv_data, kv_scale, ik_data, ik_scale, n_visible):
    """Appends T new entries per sequence ([R] 2.4.4: the main-KV latent is
    quantised after RoPE to E2M1 + E4M3/16, the indexer key to MXFP4): row t
    of sequence b goes to position n_visible[b] + t of its planes. A sequence
    whose T rows do not fit below the capacity is left unchanged. Updates the
    planes in place; returns the new visible counts.
      kv float32 [B, T, 512], ik float32 [B, T, 128] (bf16-exact values);
      planes [B, cap, 256] / [B, cap, 32] / [B, cap, 64] / [B, cap, 4] u8."""
    kv = _c(kv, np.float32)
    ik = _c(ik, np.float32)
    B, T = kv.shape[0], kv.shape[1]
    cap = kv_data.shape[1]
    out = np.array(n_visible, np.int32).copy()
    for b in range(B):
        nv = int(n_visible[b])
        if nv < 0 or nv + T > cap or T == 0:
            continue
        kv_data[b, nv:nv + T], kv_scale[b, nv:nv + T] = pack_kv_fp4(kv[b])
        ik_data[b, nv:nv + T], ik_scale[b, nv:nv + T] = quant_mxfp4(ik[b])
        out[b] = nv + T
    return out


def compress_kv(C, Z, bias, m):
    """Softmax-weighted merge of every m tokens into one entry ([V4] CSA; [B]
    4.1). C, Z [n_tokens, D], bias [m, D] -> float64 [n_tokens // m, D]."""
    C = _c(C, np.float64)
    Z = _c(Z, np.float64)
    bias = _c(bias, np.float64)
    n, D = C.shape
    out = np.zeros((n // m, D), np.float64)
    lib().orc_compress_kv(_p(C), _p(Z), _p(bias), n, m, D, _p(out))
    return out


def bf16_rne(x):
    """Round float64 values to the nearest bfloat16 value (8 significant bits,
    ties to even), returned as float64. Reading 13 of the compressor: the
    merged entry is rounded to bf16, the type of every latent the cache packs."""
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)                  # x = m 2^e, 0.5 <= |m| < 1 (m = 0 for x = 0)
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)   # np.rint: round half to even


def compress_kv_bf16(C, Z, bias, m):
    """The compressor's entries as the cache stores them: compress_kv rounded
    to bf16 (reading 13), then packed like any latent by pack_kv_fp4."""
    return bf16_rne(compress_kv(C, Z, bias, m))


def compressed_visible(pos, m):
    """Complete compressed entries visible to a query at token position pos:
    entry j covers tokens jm .. jm+m-1 and is visible once its last token is at
    or before pos."""
    j = 0
    while (j + 1) * m - 1 <= pos:
        j += 1
    return j


def main_kv_entry_bytes() -> int:
    return lib().orc_main_kv_entry_bytes()


def indexer_k_entry_bytes() -> int:
    return lib().orc_indexer_k_entry_bytes()


# ---- indexer -----------------------------------------------------------------

def index_score(q_data, q_e8m0, w, ik_data, ik_scale, n=None, positions=None):
    """Scores of one query. q_data [32,64], q_e8m0 [32,4], w [32];
    ik planes [cap,64] / [cap,4]. Scores positions 0..n-1, or `positions`.
    Returns (fp32 scores, float64 scores, multiply-accumulate count)."""
    q_data = _c(q_data, np.uint8)
    q_e8m0 = _c(q_e8m0, np.uint8)
    w = _c(w, np.float32)
    ik_data = _c(ik_data, np.uint8)
    ik_scale = _c(ik_scale, np.uint8)
    if positions is not None:
        positions = _c(positions, np.int32)
        n = positions.size
    elif n is None:
        n = ik_data.shape[0]
    out32 = np.zeros(n, np.float32)
    out64 = np.zeros(n, np.float64)
    macs = lib().orc_index_score(_p(q_data), _p(q_e8m0), _p(w), _p(ik_data), _p(ik_scale),
                                 _p(positions), n, _p(out32), _p(out64))
    return out32, out64, int(macs)


def topk(scores, k, positions=None):
    scores = _c(scores, np.float32)
    if positions is not None:
        positions = _c(positions, np.int32)
    idx = np.zeros(k, np.int32)
    nv = lib().orc_topk(_p(scores), _p(positions), scores.size, k, _p(idx))
    return idx, int(nv)


def block_pool(scores, block=8, n_blocks=2048):
    scores = _c(scores, np.float32)
    pool = np.zeros(block * n_blocks, np.int32)
    kept = lib().orc_block_pool(_p(scores), scores.size, block, n_blocks, _p(pool))
    return pool, int(kept)


def block_max(scores, block=8):
    """Block maxima of one row: [ceil(n / block)] fp32."""
    scores = _c(scores, np.float32)
    nb = (scores.size + block - 1) // block
    bmax = np.zeros(nb, np.float32)
    lib().orc_block_max(_p(scores), scores.size, block, _p(bmax))
    return bmax


def attn_merge(outs, lses):
    """outs [R, H, D], lses [R, H] (float64): the attention over the union of
    the R disjoint row sets. Returns (out [H, D], lse [H]) float64."""
    outs = _c(outs, np.float64)
    lses = _c(lses, np.float64)
    R, H, D = outs.shape
    out = np.zeros((H, D), np.float64)
    lse = np.zeros(H, np.float64)
    lib().orc_attn_merge(_p(outs), _p(lses), R, H, D, _p(out), _p(lse))
    return out, lse


def sparse_attn(q, kv_data, kv_scale, idx, swa, sm_scale=1.0):
    """q float32 [H, D] (bf16-exact values); kv planes of one sequence;
    idx int32 [k]; swa u8 [n_swa, D]. Returns (out float64 [H, D], lse [H])."""
    q = _c(q, np.float32)
    H, D = q.shape
    kv_data = _c(kv_data, np.uint8)
    kv_scale = _c(kv_scale, np.uint8)
    idx = _c(idx, np.int32)
    swa = _c(swa, np.uint8).reshape(-1, D) if swa is not None else np.zeros((0, D), np.uint8)
    out = np.zeros((H, D), np.float64)
    lse = np.zeros(H, np.float64)
    lib().orc_sparse_attn(_p(q), H, D, _p(kv_data), _p(kv_scale), _p(idx), idx.size,
                          _p(swa) if swa.size else None, swa.shape[0], float(sm_scale),
                          _p(out), _p(lse))
    return out, lse


def bounded_replay_window(i, s, W):
    """SWA positions visible to the query at position i when the SWA state is
    rebuilt by Bounded Replay from position s ([B] 6): the sliding window of
    the W most recent positions ending at i, cut at the replay start s.
    Returns the half-open range (lo, hi) of positions, lo = max(s, i - W + 1),
    hi = i + 1."""
    return max(s, i - W + 1), i + 1


def decode_batch(n_visible, q_data, q_e8m0, w, ik_data, ik_scale, kv_data, kv_scale,
                 Q, swa, k=512, sm_scale=1.0, n_threads=0):
    """Whole decode step for B sequences (score -> Top-k -> attention for the L
    layers sharing the indices). Returns (idx [B, k], out [B, L, H, D], macs)."""
    n_visible = _c(n_visible, np.int32)
    B = n_visible.size
    cap = ik_data.shape[1]
    Q = _c(Q, np.float32)
    _, L, H, D = Q.shape
    swa = _c(swa, np.uint8)
    n_swa = swa.shape[2]
    arrs = [_c(a, np.uint8) for a in (q_data, q_e8m0, ik_data, ik_scale, kv_data, kv_scale)]
    w = _c(w, np.float32)
    idx = np.zeros((B, k), np.int32)
    out = np.zeros((B, L, H, D), np.float64)
    macs = lib().orc_decode_batch(B, cap, _p(n_visible), _p(arrs[0]), _p(arrs[1]), _p(w),
                                  _p(arrs[2]), _p(arrs[3]), _p(arrs[4]), _p(arrs[5]), k, L,
                                  _p(Q), H, D, _p(swa), n_swa, float(sm_scale), _p(idx),
                                  _p(out), int(n_threads))
    return idx, out, int(macs)


def max_threads() -> int:
    return lib().orc_max_threads()
