// attention_tc.cuh -- tensor-core sparse attention partials (included by
// attention.cu, which owns g_attn_error, AttnArgs and the combine kernel).
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", section
// 2.3: each query attends to its selected main-KV entries together with the
// layer's SWA rows in one softmax; mer.dev notes section 1: 64 heads of dim
// 512 share the 512-channel latent as K and V.
//
// One CTA takes one query (64 heads) and one chunk of 128 rows (selected
// latents or SWA rows):
//   1. gather + dequantise the chunk into shared memory as bf16 R[t][c]
//      (exact: E2M1 x E4M3 has at most 6 significant bits), laid out as
//      128-byte-swizzled blocks of 64 channels;
//   2. S^T[t][h] = R[t] . Q[h] on the tensor cores (M = 128 rows, N = 64 heads,
//      K = 512; both operands K-major), accumulated in tensor memory;
//   3. per-head max and sum over the chunk's rows; P = exp(S - max) split
//      into bf16 hi + lo parts (keeps the P.V product at fp32-level accuracy);
//   4. O^T[c][h] = sum_t R[t][c] P[h][t] on the tensor cores (M = 128 channels
//      x 4 blocks, N = 64 heads, K = 128 rows), reading the same R tile as an
//      MN-major operand, once with P_hi and once with P_lo;
//   5. the unnormalised partial O and the chunk's (max, sum) per head go to the
//      workspace; attn_combine_kernel merges the chunks in fixed order.
#pragma once

#include "tc_common.cuh"

namespace csa2 {
namespace attn_tc {

constexpr int kRowsTc = 128;
constexpr int kThreads = 512;  // 16 warps: 4 TMEM lane quadrants x 4
constexpr int kOffR = 0;                                   // 8 blocks x [128 t][128 B]  = 128 KiB
constexpr int kOffQ = kOffR + kHeadDim * kRowsTc * 2;      // 8 blocks x [64 h][128 B]   =  64 KiB
constexpr int kOffP = kOffQ;  // P (2 parts x 2 blocks x [64 h][128 B] = 32 KiB) reuses Q once S^T is done
constexpr int kPBytes = kHeads * kRowsTc * 2;              // 16 KiB per P part
constexpr int kOffMisc = kOffQ + kHeadDim * kHeads * 2;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;      // S^T: 64 columns (heads), lanes = rows
constexpr uint32_t kColO = 64;     // O^T: 4 blocks x 64 columns, lanes = channels

static_assert(kSmemBytes <= 232448, "shared memory budget");

// exact bf16x2 product (operands with <= 2 and <= 4 significant bits)
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Four E2M1 codes (the 16-bit x: channel i in bits 4i..4i+3) to four exact
// bf16 values in two bf16x2 words, in registers: the magnitudes come from two
// 8-entry byte tables (low and high byte of the bf16 of 0, 0.5, 1, 1.5, 2, 3,
// 4, 6) picked by prmt, the signs from a sign-replicating prmt.
__device__ __forceinline__ void e2m1x4_to_bf16(uint32_t x, uint32_t& v01, uint32_t& v23) {
  constexpr uint32_t kLoA = 0xC0800000u, kLoB = 0xC0804000u;  // low bytes, magnitudes 0..3 and 4..7
  constexpr uint32_t kHiA = 0x3F3F3F00u, kHiB = 0x40404040u;  // high bytes
  const uint32_t sel = x & 0x7777u;
  const uint32_t lo4 = __byte_perm(kLoA, kLoB, sel);
  uint32_t hi4 = __byte_perm(kHiA, kHiB, sel);
  // msb of bytes: x << 4 holds the signs of channels 0 and 2, x those of 1 and 3
  uint32_t smask;
  asm("prmt.b32 %0, %1, %2, 0x9D8C;" : "=r"(smask) : "r"(x), "r"(x << 4));
  hi4 |= smask & 0x80808080u;
  v01 = __byte_perm(lo4, hi4, 0x5140);
  v23 = __byte_perm(lo4, hi4, 0x7362);
}

// Transpose-reduce across a warp: lane L holds v[0..N) (one value per head,
// N = 16 or 32); afterwards lane L returns the reduction over all 32 lanes of
// head L mod N. Each stage halves the values a lane keeps (N/2 + ... + 1
// shuffles); for N = 16 a last shuffle joins the two half-warps. v is
// overwritten.
template <bool kMax, int N>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[N], int lane) {
#pragma unroll
  for (int width = N / 2; width >= 1; width >>= 1) {
    const bool up = (lane & width) != 0;
#pragma unroll
    for (int i = 0; i < width; ++i) {
      const float keep = up ? v[i + width] : v[i];
      const float send = up ? v[i] : v[i + width];
      const float got = __shfl_xor_sync(0xffffffffu, send, width);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  float r = v[0];
  if (N == 16) {
    const float o = __shfl_xor_sync(0xffffffffu, r, 16);
    r = kMax ? fmaxf(r, o) : r + o;
  }
  return r;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_partial_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, AttnArgs a) {
  pdl_begin();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = tc::smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  uint8_t* sR = sm + kOffR;
  uint8_t* sQ = sm + kOffQ;
  uint8_t* sP = sm + kOffP;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kOffMisc);
  uint64_t* q_bar = bar + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + kOffMisc + 16);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + kOffMisc + 20);
  __shared__ float red[4][kHeads];
  __shared__ float m_s[kHeads], l_s[kHeads];
  __shared__ uint16_t lut_e4m3[256];   // E4M3 byte -> bf16 value
  __shared__ int row_valid[kRowsTc];  // 0 none, 1 selected latent, 2 SWA row
  __shared__ int64_t row_src[kRowsTc];  // entry index in the plane, or SWA byte offset

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lq = blockIdx.y;
  const int qi = a.q0 + lq;
  const int seq = qi / a.L;
  const int split = blockIdx.x;

  // ---- Q: [64 h][512 c] bf16 -> 8 TMA boxes of [64 h][64 c] = [64][128 B], SW128 ----
  if (tid == 0) {
    tc::mbar_init(bar, 1);
    tc::mbar_init(q_bar, 1);
    *s_abort = 0;
    tc::fence_mbar_init();
    tc::mbar_arrive_expect_tx(q_bar, kHeads * kHeadDim * 2);
    for (int blk = 0; blk < kHeadDim / 64; ++blk)
      tc::tma_load_2d(sQ + blk * (kHeads * 128), &tmap_q, blk * 64, qi * kHeads, q_bar);
  }
  if (warp == 0) tc::tmem_alloc(s_tmem, kTmemCols);
  if (tid < 256) {
    const uint32_t byte = (uint32_t)tid;
    __nv_bfloat16 e = __float2bfloat16_rn(e4m3_to_f32(byte));  // exact (4 significant bits)
    lut_e4m3[byte] = *reinterpret_cast<uint16_t*>(&e);
  }
  // ---- rows of this chunk: position (or SWA row), validity ----
  const int64_t nv = a.n_visible ? (int64_t)a.n_visible[seq] : a.nv_const;
  const int32_t* idx_row = a.idx + (int64_t)seq * a.k;
  if (tid < kRowsTc) {
    const int t = split * kRowsTc + tid;
    int valid = 0;
    int64_t src = 0;
    if (t < a.k) {
      const int32_t p = idx_row[t];
      if (p >= 0) {
        if (p < nv) {
          valid = 1;                                   // selected latent
          src = (int64_t)seq * a.kv_seq_stride + p;
        } else {
          record_error(&g_attn_error, CSA2_ERR_DEVICE);
        }
      }
    } else if (t < a.k + a.n_swa) {
      valid = 2;                                       // SWA row
      src = (int64_t)qi * a.swa_q_stride + (int64_t)(t - a.k) * kHeadDim;
    }
    row_valid[tid] = valid;
    row_src[tid] = src;
  }
  __syncthreads();
  // ---- gather + dequantise R: [128 t][512 c] bf16 as 8 blocks [128 t][128 B] ----
  // warp w owns rows 8w..8w+7; pass j covers them in 64-channel block j, 4
  // lanes per row, each lane 16 channels (two 16-byte chunks). All loads of a
  // thread are issued before any is used.
  {
    constexpr int kPasses = 8;
    uint4 raw[kPasses];
    uint32_t sc[kPasses];
#pragma unroll
    for (int jj = 0; jj < kPasses; ++jj) {
      const int r = warp * 8 + (lane >> 2);
      const int blk = jj * 4 + (lane & 3);
      const int kind = row_valid[r];
      const int64_t src = row_src[r];
      raw[jj] = make_uint4(0u, 0u, 0u, 0u);
      sc[jj] = 0u;
      if (kind == 1) {
        const uint2 v = *reinterpret_cast<const uint2*>(a.kv_data + src * kKvBytes + blk * 8);
        raw[jj].x = v.x;
        raw[jj].y = v.y;
        sc[jj] = a.kv_scale[src * kKvScales + blk];
      } else if (kind == 2) {
        raw[jj] = *reinterpret_cast<const uint4*>(a.swa + src + blk * 16);
      }
    }
#pragma unroll
    for (int jj = 0; jj < kPasses; ++jj) {
      const int r = warp * 8 + (lane >> 2);
      const int blk = jj * 4 + (lane & 3);
      const int kind = row_valid[r];
      uint32_t o[8];
      if (kind == 1) {
        const uint32_t s1 = lut_e4m3[sc[jj]];
        const uint32_t s2 = s1 | (s1 << 16);
        const uint32_t w[2] = {raw[jj].x, raw[jj].y};
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          uint32_t v01, v23;
          e2m1x4_to_bf16((w[e >> 2] >> (8 * (e & 3))) & 0xFFFFu, v01, v23);
          o[e] = mul_bf16x2(v01, s2);
          o[e + 1] = mul_bf16x2(v23, s2);
        }
      } else {
        const uint32_t w[4] = {raw[jj].x, raw[jj].y, raw[jj].z, raw[jj].w};  // zero for invalid rows
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t pair = w[e >> 1] >> (16 * (e & 1));
          o[e] = (uint32_t)lut_e4m3[pair & 0xFFu] | ((uint32_t)lut_e4m3[(pair >> 8) & 0xFFu] << 16);
        }
      }
      uint8_t* region = sR + (blk >> 2) * (kRowsTc * 128);
      const uint32_t c0 = (uint32_t)(blk & 3) * 2;
      *reinterpret_cast<uint4*>(region + tc::sw128_offset(r, c0)) = make_uint4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<uint4*>(region + tc::sw128_offset(r, c0 + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;

  // ---- S^T = R . Q^T : M = 128 rows, N = 64 heads, K = 512 ----
  bool q_ok = tc::mbar_wait_bounded(q_bar, 0, s_abort, &g_attn_error);
  if (tid == 0 && q_ok) {
    constexpr uint32_t idesc = tc::idesc_bf16(128, 64, 0, 0);
    const uint32_t r_addr = tc::smem_u32(sR), q_addr = tc::smem_u32(sQ);
    for (int kk = 0; kk < kHeadDim / 16; ++kk) {
      const uint32_t blk = (uint32_t)kk >> 2, off = ((uint32_t)kk & 3u) * 32u;
      const uint64_t ad = tc::smem_desc(r_addr + blk * (kRowsTc * 128) + off, 0, 1024, tc::kSwizzle128B);
      const uint64_t bd = tc::smem_desc(q_addr + blk * (kHeads * 128) + off, 0, 1024, tc::kSwizzle128B);
      tc::mma_bf16(tmem + kColS, ad, bd, idesc, kk > 0 ? 1u : 0u);
    }
    tc::mma_commit(bar);
  }
  __syncwarp();
  // warp-uniform outcomes: the tcgen05.ld below needs the whole warp
  bool ok = __all_sync(0xffffffffu, tc::mbar_wait_bounded(bar, 0, s_abort, &g_attn_error));
  tc::tc_fence_after();

  // ---- softmax over the chunk's rows; warp w: rows 32*(w%4).., heads 16*(w/4).. ----
  constexpr int kHpw = 16;  // heads per warp
  const int rq = warp & 3, hb = (warp >> 2) * kHpw;
  const int row = rq * 32 + lane;
  const bool rv = ok && row_valid[row] != 0;
  const uint32_t s_addr = tmem + ((uint32_t)(rq * 32) << 16) + kColS + hb;
  float p[kHpw];
  auto load_scores = [&]() {
    uint32_t r[kHpw];
    if (ok) {
      tc::tmem_ld_32x32b_x16(s_addr, r);
      tc::tmem_ld_wait();
    }
#pragma unroll
    for (int j = 0; j < kHpw; ++j) p[j] = rv ? __uint_as_float(r[j]) * a.sm_scale : -INFINITY;
  };
  load_scores();
  // per-head max over the warp's 32 rows lands in lane (head - hb) mod 16
  {
    const float m = warp_transpose_reduce<true, kHpw>(p, lane);
    if (lane < kHpw) red[rq][hb + lane] = m;
  }
  __syncthreads();
  if (tid < kHeads) m_s[tid] = fmaxf(fmaxf(red[0][tid], red[1][tid]), fmaxf(red[2][tid], red[3][tid]));
  __syncthreads();
  // P = exp(S - m) from a second read of S; P_hi = bf16(P), P_lo = bf16(P - P_hi)
  load_scores();
#pragma unroll
  for (int j = 0; j < kHpw; ++j) p[j] = (p[j] == -INFINITY) ? 0.0f : expf(p[j] - m_s[hb + j]);
  // P parts, K-major for the PV MMA: [64 h][128 t] as 2 blocks of [64 h][128 B]
  {
    uint8_t* blkp = sP + (row >> 6) * (kHeads * 128);
    const uint32_t chunk = (uint32_t)(row & 63) >> 3, within = ((uint32_t)row & 7u) * 2u;
#pragma unroll
    for (int j = 0; j < kHpw; ++j) {
      const int h = hb + j;
      const __nv_bfloat16 hi = __float2bfloat16_rn(p[j]);
      const __nv_bfloat16 lo = __float2bfloat16_rn(p[j] - __bfloat162float(hi));
      const uint32_t off = tc::sw128_offset((uint32_t)h, chunk) + within;
      *reinterpret_cast<__nv_bfloat16*>(blkp + off) = hi;
      *reinterpret_cast<__nv_bfloat16*>(blkp + kPBytes + off) = lo;
    }
  }
  __syncthreads();  // red[] reads for m_s are done before it is reused for the sums
  {
    const float l = warp_transpose_reduce<false, kHpw>(p, lane);
    if (lane < kHpw) red[rq][hb + lane] = l;
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (tid < kHeads) l_s[tid] = red[0][tid] + red[1][tid] + red[2][tid] + red[3][tid];

  // ---- O^T = R^T . P^T : 4 x (M = 128 channels), N = 64 heads, K = 128 rows ----
  if (tid == 0 && ok) {
    constexpr uint32_t idesc = tc::idesc_bf16(128, 64, 1, 0);  // A (channels x rows) is MN-major
    const uint32_t r_addr = tc::smem_u32(sR), p_addr = tc::smem_u32(sP);
    for (int mb = 0; mb < 4; ++mb) {
      for (int part = 0; part < 2; ++part) {
        for (int kk = 0; kk < kRowsTc / 16; ++kk) {
          // A: channels 128*mb .. +127 (64-channel blocks 2mb, 2mb+1: LBO apart),
          //    rows 16*kk .. +15 (8-row groups: SBO apart)
          const uint64_t ad = tc::smem_desc(r_addr + (uint32_t)(2 * mb) * (kRowsTc * 128) + (uint32_t)kk * 16u * 128u,
                                            kRowsTc * 128, 1024, tc::kSwizzle128B);
          // B: P part, heads 0..63, rows 16*kk .. +15 (64-row K blocks of 128 B)
          const uint64_t bd = tc::smem_desc(p_addr + (uint32_t)part * kPBytes + (uint32_t)(kk >> 2) * (kHeads * 128) +
                                                ((uint32_t)kk & 3u) * 32u,
                                            0, 1024, tc::kSwizzle128B);
          tc::mma_bf16(tmem + kColO + 64u * (uint32_t)mb, ad, bd, idesc, (part | kk) ? 1u : 0u);
        }
      }
    }
    tc::mma_commit(bar);
  }
  __syncwarp();
  ok = __all_sync(0xffffffffu, ok && tc::mbar_wait_bounded(bar, 1, s_abort, &g_attn_error));
  tc::tc_fence_after();

  // ---- partial O (unnormalised, fp32) and (max, sum) to the workspace ----
  float* po = a.part_o + ((int64_t)lq * a.n_split + split) * kHeads * kHeadDim;
  if (ok) {
    // warp w: channel lanes of quadrant w%4, channel block mb = w/4
    for (int mbi = 0; mbi < 1; ++mbi) {
      const int mb = warp >> 2;
      const int c = mb * 128 + rq * 32 + lane;
      for (int hh = 0; hh < kHeads; hh += 32) {
        uint32_t r[32];
        tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(rq * 32) << 16) + kColO + 64u * (uint32_t)mb + (uint32_t)hh, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) po[(hh + j) * kHeadDim + c] = __uint_as_float(r[j]);
      }
    }
  }
  if (tid < kHeads) {
    float* ml = a.part_ml + (((int64_t)lq * a.n_split + split) * kHeads + tid) * 2;
    ml[0] = m_s[tid];
    ml[1] = ok ? l_s[tid] : 0.0f;
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace attn_tc
}  // namespace csa2
