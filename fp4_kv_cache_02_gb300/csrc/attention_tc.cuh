// attention_tc.cuh -- tensor-core sparse attention partials (included by
// attention.cu, which owns g_attn_error, AttnArgs and the combine kernel).
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", section
// 2.3: each query attends to its selected main-KV entries together with the
// layer's SWA rows in one softmax; mer.dev notes section 1: 64 heads of dim
// 512 share the 512-channel latent as K and V.
//
// One CTA takes one query (64 heads) and one chunk of `rows` rows (selected
// latents and/or SWA rows; rows is a multiple of 32, at most 160, chosen by
// the host so that the grid fills the SMs in as few waves as possible):
//   1. all row loads are issued up front; the chunk is dequantised into
//      shared memory as bf16 R[t][c] (exact: E2M1 x E4M3 has at most 6
//      significant bits) in 128-byte-swizzled blocks of 64 channels, the low
//      256 channels first;
//   2. S^T[t][h] = R[t] . Q[h] on the tensor cores (M = 128 rows per tile, one
//      or two tiles; N = 64 heads; K = 512 in quarters of 128 channels held
//      in three slots: quarter 3 loads into quarter 0's slot once its MMAs are
//      done, while the high channels are dequantised);
//   3. per-head max and sum over the chunk's rows; P = exp(S - max) split
//      into bf16 hi + lo parts (keeps the P.V product at fp32-level accuracy),
//      stacked as 128 B-operand rows (64 hi, 64 lo);
//   4. O^T[c][n] = sum_t R[t][c] P[n][t] on the tensor cores (M = 128 channels
//      x 4 blocks, N = 128, K = rows), reading the same R tile as an MN-major
//      operand; O = O_hi + O_lo when read back;
//   5. the chunks of a query merge: when they form one thread-block cluster
//      (at most 8 chunks) each scales its O by exp(m - M) / L into its shared
//      memory and each rank sums a slice of the heads over the cluster in rank
//      order through distributed shared memory, writing the output directly;
//      otherwise the unnormalised partial O and (max, sum) go to the workspace
//      and attn_combine_kernel merges the chunks in the same fixed order.
#pragma once

#include "tc_common.cuh"

namespace csa2 {
namespace attn_tc {

constexpr int kMaxRows = 160;   // rows per CTA: a multiple of 32, at most 160
constexpr int kMaxClusterChunks = 8;  // chunks of a query merged inside one cluster
constexpr int kThreads = 512;   // 16 warps: 4 TMEM lane quadrants x 4
constexpr int kBlkR = kMaxRows * 128;                     // one 64-channel block of R: [160 t][128 B]
constexpr int kOffR = 0;                                  // 8 blocks                        = 160 KiB
constexpr int kOffQP = kOffR + 8 * kBlkR;                 // Q half (4 x [64 h][128 B]) or P = 48 KiB
constexpr int kQQuarterBytes = kHeads * 128 * 2;          // 16 KiB: channels 128q .. 128q+127
constexpr int kPBlk = 2 * kHeads * 128;                   // P: per 64 rows, [128 n][128 B]  = 16 KiB
constexpr int kOffMisc = kOffQP + 3 * kPBlk;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;      // S^T: tile t at columns 64t .. 64t+63 (heads), lanes = rows
constexpr uint32_t kColO = 0;      // O^T: 4 blocks x 128 columns (64 hi + 64 lo), lanes = channels;
                                   // written once S^T has been read

static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(3 * kQQuarterBytes <= 3 * kPBlk, "three Q quarters fit the P region");

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
  // barriers, tensor memory and the E4M3 table need nothing from the preceding
  // kernel; its outputs (the indices, possibly Q) are read after pdl_wait()
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = tc::smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  uint8_t* sR = sm + kOffR;
  uint8_t* sQP = sm + kOffQP;
  uint64_t* bar_s0 = reinterpret_cast<uint64_t*>(sm + kOffMisc);  // S^T over channels 0..127 done
  uint64_t* bar_s1 = bar_s0 + 1;                                 // S^T complete
  uint64_t* bar_pv = bar_s0 + 2;                                 // O^T complete
  uint64_t* q_full = bar_s0 + 3;                                 // 3 Q slots (slot 0 twice)
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + kOffMisc + 48);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + kOffMisc + 52);
  __shared__ float red[4][kHeads];
  __shared__ float m_s[kHeads], l_s[kHeads];
  __shared__ uint16_t lut_e4m3[256];     // E4M3 byte -> bf16 value
  __shared__ int row_valid[kMaxRows];    // 0 none, 1 selected latent, 2 SWA row
  __shared__ int64_t row_src[kMaxRows];  // entry index in the plane, or SWA byte offset

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lq = blockIdx.y;
  const int qi = a.q0 + lq;
  const int seq = qi / a.L;
  const int split = blockIdx.x;
  const int rows = a.rows;
  const int n_tiles = (rows + 127) >> 7;

  // ---- Q channels 0..255: 4 TMA boxes of [64 h][64 c] = [64][128 B], SW128 ----
  if (tid == 0) {
    tc::mbar_init(bar_s0, 1);
    tc::mbar_init(bar_s1, 1);
    tc::mbar_init(bar_pv, 1);
    for (int q = 0; q < 3; ++q) tc::mbar_init(&q_full[q], 1);
    *s_abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(s_tmem, kTmemCols);
  if (tid < 256) {
    const uint32_t byte = (uint32_t)tid;
    __nv_bfloat16 e = __float2bfloat16_rn(e4m3_to_f32(byte));  // exact (4 significant bits)
    lut_e4m3[byte] = *reinterpret_cast<uint16_t*>(&e);
  }
  pdl_wait();
  // Q quarter q (channels 128q .. +127, two boxes of [64 h][64 c]) into slot
  // q % 3 of the Q/P region: quarters 0-2 now, quarter 3 once quarter 0's
  // MMAs have read slot 0
  auto load_q_quarter = [&](const int q) {
    uint8_t* slot = sQP + (q % 3) * kQQuarterBytes;
    tc::mbar_arrive_expect_tx(&q_full[q % 3], kQQuarterBytes);
    for (int blk = 0; blk < 2; ++blk)
      tc::tma_load_2d(slot + blk * (kHeads * 128), &tmap_q, q * 128 + blk * 64, qi * kHeads, &q_full[q % 3]);
  };
  if (tid == 0)
    for (int q = 0; q < 3; ++q) load_q_quarter(q);
  // ---- rows of this chunk: position (or SWA row), validity ----
  const int64_t nv = a.n_visible ? (int64_t)a.n_visible[seq] : a.nv_const;
  const int32_t* idx_row = a.idx + (int64_t)seq * a.k;
  if (tid < rows) {
    const int t = split * rows + tid;
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
      // SWA row; in prefill row j of query qi is row qi + j of the array, and
      // rows before swa_first_row lie before a Bounded Replay start
      if ((int64_t)qi + (t - a.k) >= (int64_t)a.swa_first_row) {
        valid = 2;
        src = (int64_t)qi * a.swa_q_stride + (int64_t)(t - a.k) * kHeadDim;
      }
    }
    row_valid[tid] = valid;
    row_src[tid] = src;
  }
  __syncthreads();

  // ---- gather: all loads first. Pass ps covers rows 64ps .. 64ps+63: warp w
  // rows 64ps + 4w .. +3, 8 lanes per row; lane `sub` holds channels
  // 32sub .. 32sub+31 of the low half and of the high half of the row ----
  constexpr int kPasses = (kMaxRows + 63) / 64;
  const int grp = lane >> 3, sub = lane & 7;
  uint4 raw[kPasses][4];
#pragma unroll
  for (int ps = 0; ps < kPasses; ++ps) {
    const int r = ps * 64 + warp * 4 + grp;
    const int kind = r < rows ? row_valid[r] : 0;
    const int64_t src = r < rows ? row_src[r] : 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) raw[ps][i] = make_uint4(0u, 0u, 0u, 0u);
    if (kind == 1) {
      const uint8_t* d = a.kv_data + src * kKvBytes + sub * 16;
      raw[ps][0] = *reinterpret_cast<const uint4*>(d);
      raw[ps][1] = *reinterpret_cast<const uint4*>(d + 128);
      const uint8_t* sc = a.kv_scale + src * kKvScales + sub * 2;
      raw[ps][2].x = (uint32_t)*reinterpret_cast<const uint16_t*>(sc) |
                     ((uint32_t)*reinterpret_cast<const uint16_t*>(sc + 16) << 16);
    } else if (kind == 2) {
      const uint8_t* e = a.swa + src + sub * 32;
      raw[ps][0] = *reinterpret_cast<const uint4*>(e);
      raw[ps][1] = *reinterpret_cast<const uint4*>(e + 16);
      raw[ps][2] = *reinterpret_cast<const uint4*>(e + 256);
      raw[ps][3] = *reinterpret_cast<const uint4*>(e + 272);
    }
  }
  // dequantise one half (channels 256h .. 256h+255) of every row into R
  auto dequant_half = [&](const int half) {
#pragma unroll
    for (int ps = 0; ps < kPasses; ++ps) {
      const int r = ps * 64 + warp * 4 + grp;
      if (r >= rows) continue;
      const int kind = row_valid[r];
      uint32_t o[16];
      if (kind == 1) {
        const uint4 d = raw[ps][half];
        const uint32_t scb = (raw[ps][2].x >> (16 * half)) & 0xFFFFu;
        const uint32_t sa = lut_e4m3[scb & 0xFFu], sb = lut_e4m3[scb >> 8];
        const uint32_t sa2 = sa | (sa << 16), sb2 = sb | (sb << 16);
        const uint32_t w[4] = {d.x, d.y, d.z, d.w};  // w[i]: channels 8i .. 8i+7 of the lane's 32
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t v01, v23;
            e2m1x4_to_bf16((w[i] >> (16 * hh)) & 0xFFFFu, v01, v23);
            const uint32_t s2 = i < 2 ? sa2 : sb2;   // channels 0..15: scale a, 16..31: scale b
            o[4 * i + 2 * hh] = mul_bf16x2(v01, s2);
            o[4 * i + 2 * hh + 1] = mul_bf16x2(v23, s2);
          }
        }
      } else if (kind == 2) {
        const uint4 x = raw[ps][2 * half], y = raw[ps][2 * half + 1];
        const uint32_t w[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint32_t pair = w[e >> 1] >> (16 * (e & 1));
          o[e] = (uint32_t)lut_e4m3[pair & 0xFFu] | ((uint32_t)lut_e4m3[(pair >> 8) & 0xFFu] << 16);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) o[e] = 0u;   // invalid rows are zero: P = 0 must not meet NaN
      }
      uint8_t* region = sR + (half * 4 + (sub >> 1)) * kBlkR;
      const uint32_t c0 = (uint32_t)(sub & 1) * 4;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(region + tc::sw128_offset((uint32_t)r, c0 + j)) =
            make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
    }
  };
  // S^T (+)= R[:, 128q .. +127] . Q[:, 128q .. +127]^T for every tile of 128 rows
  auto issue_s = [&](const uint32_t tmem, const int q) {
    constexpr uint32_t idesc = tc::idesc_bf16(128, 64, 0, 0);
    const uint32_t r_addr = tc::smem_u32(sR), q_addr = tc::smem_u32(sQP) + (uint32_t)((q % 3) * kQQuarterBytes);
    for (int t = 0; t < n_tiles; ++t)
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t blk = (uint32_t)(q * 2) + ((uint32_t)kk >> 2), off = ((uint32_t)kk & 3u) * 32u;
        const uint64_t ad = tc::smem_desc(r_addr + blk * kBlkR + (uint32_t)t * (128u * 128u) + off, 0, 1024,
                                          tc::kSwizzle128B);
        const uint64_t bd = tc::smem_desc(q_addr + ((uint32_t)kk >> 2) * (kHeads * 128) + off, 0, 1024,
                                          tc::kSwizzle128B);
        tc::mma_bf16(tmem + kColS + 64u * (uint32_t)t, ad, bd, idesc, (q | kk) ? 1u : 0u);
      }
  };

  dequant_half(0);
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  bool lead_ok = true;   // meaningful in thread 0
  if (tid == 0) {
    lead_ok = tc::mbar_wait_bounded(&q_full[0], 0, s_abort, &g_attn_error);
    if (lead_ok) {
      issue_s(tmem, 0);
      tc::mma_commit(bar_s0);
      lead_ok = tc::mbar_wait_bounded(&q_full[1], 0, s_abort, &g_attn_error);
      if (lead_ok) issue_s(tmem, 1);
    }
  }
  dequant_half(1);
  if (tid == 0 && lead_ok) {
    // slot 0 takes quarter 3 once quarter 0's MMAs have read it
    lead_ok = tc::mbar_wait_bounded(bar_s0, 0, s_abort, &g_attn_error);
    if (lead_ok) load_q_quarter(3);
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (tid == 0 && lead_ok) {
    lead_ok = tc::mbar_wait_bounded(&q_full[2], 0, s_abort, &g_attn_error);
    if (lead_ok) {
      issue_s(tmem, 2);
      lead_ok = tc::mbar_wait_bounded(&q_full[0], 1, s_abort, &g_attn_error);
      if (lead_ok) {
        issue_s(tmem, 3);
        tc::mma_commit(bar_s1);
      }
    }
  }
  if (tid == 0 && !lead_ok) *s_abort = 1;
  __syncwarp();
  // warp-uniform outcomes: the tcgen05.ld below needs the whole warp
  const bool s_ok = __all_sync(0xffffffffu, tc::mbar_wait_bounded(bar_s1, 0, s_abort, &g_attn_error));
  tc::tc_fence_after();

  // ---- softmax over the chunk's rows. Warp w reads TMEM lanes 32(w%4) .. (rows
  // 32(w%4) + lane of tile 0, and rows 128 + lane of tile 1 for w%4 == 0) and
  // heads 16(w/4) .. +15 ----
  constexpr int kHpw = 16;  // heads per warp
  const int rq = warp & 3, hb = (warp >> 2) * kHpw;
  const int row0 = rq * 32 + lane, row1 = 128 + lane;
  const bool two = n_tiles > 1 && rq == 0;  // warp-uniform
  const bool rv0 = s_ok && row0 < rows && row_valid[row0] != 0;
  const bool rv1 = s_ok && two && row1 < rows && row_valid[row1] != 0;
  float p0[kHpw], p1[kHpw];
  auto load_scores = [&]() {
    uint32_t r0[kHpw], r1[kHpw];
    if (s_ok) {
      tc::tmem_ld_32x32b_x16(tmem + ((uint32_t)(rq * 32) << 16) + kColS + hb, r0);
      if (two) tc::tmem_ld_32x32b_x16(tmem + kColS + 64u + hb, r1);
      tc::tmem_ld_wait();
    }
#pragma unroll
    for (int j = 0; j < kHpw; ++j) {
      p0[j] = rv0 ? __uint_as_float(r0[j]) * a.sm_scale : -INFINITY;
      p1[j] = rv1 ? __uint_as_float(r1[j]) * a.sm_scale : -INFINITY;
    }
  };
  load_scores();
  // per-head max over the warp's rows lands in lane (head - hb) mod 16
  {
    float v[kHpw];
#pragma unroll
    for (int j = 0; j < kHpw; ++j) v[j] = fmaxf(p0[j], p1[j]);
    const float m = warp_transpose_reduce<true, kHpw>(v, lane);
    if (lane < kHpw) red[rq][hb + lane] = m;
  }
  __syncthreads();
  if (tid < kHeads) m_s[tid] = fmaxf(fmaxf(red[0][tid], red[1][tid]), fmaxf(red[2][tid], red[3][tid]));
  __syncthreads();
  // P = exp(S - m) from a second read of S; P_hi = bf16(P), P_lo = bf16(P - P_hi),
  // stored K-major for the PV MMA as B-operand rows n = h (hi) and 64 + h (lo):
  // per 64 rows t a block of [128 n][128 B]
  // the scores are still in p0 / p1 (the reduction worked on a copy);
  // exp(s - m) = 2^(s log2 e - m log2 e); only the warps of lane quadrant 0
  // hold rows of the second tile
  constexpr float kLog2e = 1.4426950408889634f;
#pragma unroll
  for (int j = 0; j < kHpw; ++j) {
    const float ml = m_s[hb + j] * kLog2e;
    p0[j] = (p0[j] == -INFINITY) ? 0.0f : exp2f(fmaf(p0[j], kLog2e, -ml));
  }
  if (two) {
#pragma unroll
    for (int j = 0; j < kHpw; ++j) {
      const float ml = m_s[hb + j] * kLog2e;
      p1[j] = (p1[j] == -INFINITY) ? 0.0f : exp2f(fmaf(p1[j], kLog2e, -ml));
    }
  } else {
#pragma unroll
    for (int j = 0; j < kHpw; ++j) p1[j] = 0.0f;
  }
  auto store_p = [&](const int t, const float (&pv)[kHpw]) {
    uint8_t* blkp = sQP + (t >> 6) * kPBlk;
    const uint32_t chunk = (uint32_t)(t & 63) >> 3, within = ((uint32_t)t & 7u) * 2u;
#pragma unroll
    for (int j = 0; j < kHpw; ++j) {
      const uint32_t h = (uint32_t)(hb + j);
      const __nv_bfloat16 hi = __float2bfloat16_rn(pv[j]);
      const __nv_bfloat16 lo = __float2bfloat16_rn(pv[j] - __bfloat162float(hi));
      *reinterpret_cast<__nv_bfloat16*>(blkp + tc::sw128_offset(h, chunk) + within) = hi;
      *reinterpret_cast<__nv_bfloat16*>(blkp + tc::sw128_offset(h + kHeads, chunk) + within) = lo;
    }
  };
  if (row0 < rows) store_p(row0, p0);
  if (two && row1 < rows) store_p(row1, p1);
  __syncthreads();  // red[] reads for m_s are done before it is reused for the sums
  {
    float v[kHpw];
#pragma unroll
    for (int j = 0; j < kHpw; ++j) v[j] = p0[j] + p1[j];
    const float l = warp_transpose_reduce<false, kHpw>(v, lane);
    if (lane < kHpw) red[rq][hb + lane] = l;
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (tid < kHeads) l_s[tid] = red[0][tid] + red[1][tid] + red[2][tid] + red[3][tid];

  // ---- O^T = R^T . [P_hi; P_lo]^T : 4 x (M = 128 channels), N = 128, K = rows ----
  if (tid == 0 && s_ok) {
    constexpr uint32_t idesc = tc::idesc_bf16(128, 128, 1, 0);  // A (channels x rows) is MN-major
    const uint32_t r_addr = tc::smem_u32(sR), p_addr = tc::smem_u32(sQP);
    const int ksteps = rows / 16;
    for (int mb = 0; mb < 4; ++mb) {
      for (int kk = 0; kk < ksteps; ++kk) {
        // A: channels 128mb .. +127 (64-channel blocks 2mb, 2mb+1: LBO apart),
        //    rows 16kk .. +15 (8-row groups: SBO apart)
        const uint64_t ad = tc::smem_desc(r_addr + (uint32_t)(2 * mb) * kBlkR + (uint32_t)kk * 16u * 128u, kBlkR,
                                          1024, tc::kSwizzle128B);
        // B: 128 P rows (hi, lo), rows t = 16kk .. +15 inside the 64-row block kk/4
        const uint64_t bd = tc::smem_desc(p_addr + (uint32_t)(kk >> 2) * kPBlk + ((uint32_t)kk & 3u) * 32u, 0, 1024,
                                          tc::kSwizzle128B);
        tc::mma_bf16(tmem + kColO + 128u * (uint32_t)mb, ad, bd, idesc, kk ? 1u : 0u);
      }
    }
    tc::mma_commit(bar_pv);
  }
  __syncwarp();
  const bool ok = __all_sync(0xffffffffu, s_ok && tc::mbar_wait_bounded(bar_pv, 0, s_abort, &g_attn_error));
  tc::tc_fence_after();

  // warp w reads the O^T lanes of quadrant w%4 in channel block mb = w/4
  const int mb = warp >> 2;
  const int c_own = mb * 128 + rq * 32 + lane;
  const uint32_t o_base = tmem + ((uint32_t)(rq * 32) << 16) + kColO + 128u * (uint32_t)mb;
  if (a.fused) {
    // ---- merge inside the cluster of this query's chunks (rank = split) ----
    // each chunk stores its unnormalised O as [h][c] fp32 in its own shared
    // memory; after one cluster barrier every CTA reads all chunks' (m, l),
    // forms the weights exp(m_j - M) / L, and rank r sums heads
    // [64r/n, 64(r+1)/n) over the chunks in fixed order, writing the output.
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    const int nsp = a.n_split;
    const int rank = (int)cl.block_rank();
    __shared__ float w_s[kMaxClusterChunks][kHeads];   // m_j, then the weights
    __shared__ float f_l[kMaxClusterChunks][kHeads];   // l_j, then l_j exp(m_j - M)
    __shared__ float e_s[kMaxClusterChunks][kHeads];   // exp(m_j - M)
    __shared__ float M_s[kHeads];
    float* o_s = reinterpret_cast<float*>(sR);  // 128 KiB of the R tile, free after the PV product
#pragma unroll
    for (int hh = 0; hh < kHeads; hh += 32) {
      uint32_t rh[32], rl[32];
      if (ok) {
        tc::tmem_ld_32x32b_x32(o_base + (uint32_t)hh, rh);
        tc::tmem_ld_32x32b_x32(o_base + (uint32_t)(kHeads + hh), rl);
        tc::tmem_ld_wait();
      }
#pragma unroll
      for (int j = 0; j < 32; ++j)
        o_s[(hh + j) * kHeadDim + c_own] = ok ? __uint_as_float(rh[j]) + __uint_as_float(rl[j]) : 0.0f;
    }
    if (tid < kHeads && !ok) l_s[tid] = 0.0f;
    cl.sync();
    // rank r sums heads [64r/n, 64(r+1)/n): items i = tid + kThreads u are
    // float4 columns of that slice; the remote loads of the first two items
    // go out before the weights are formed
    const int h0 = kHeads * rank / nsp, h1 = kHeads * (rank + 1) / nsp;
    const int n_items = (h1 - h0) * (kHeadDim / 4);
    float4 v[2][kMaxClusterChunks];
    auto load_items = [&](const int i0) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int i = i0 + u * kThreads;
        const int h = h0 + i / (kHeadDim / 4), c4 = (i % (kHeadDim / 4)) * 4;
#pragma unroll
        for (int j = 0; j < kMaxClusterChunks; ++j)
          if (j < nsp && i < n_items)
            v[u][j] = *reinterpret_cast<const float4*>(cl.map_shared_rank(o_s, j) + h * kHeadDim + c4);
      }
    };
    load_items(tid);
    // (m, l) of every chunk, one remote load each; e_j = l_j exp(m_j - M)
    if (tid < nsp * kHeads) {
      const int j = tid / kHeads, h = tid % kHeads;
      const float lj = *cl.map_shared_rank(&l_s[h], j);
      w_s[j][h] = lj > 0.0f ? *cl.map_shared_rank(&m_s[h], j) : -INFINITY;
      f_l[j][h] = lj;
    }
    __syncthreads();
    // thread (j, h): M = max_j m_j, e_j = exp(m_j - M), then L = sum_j l_j e_j in
    // fixed order and the weight e_j / L (m_s and l_s stay as they are: the
    // other CTAs of the cluster may still be reading them)
    if (tid < nsp * kHeads) {
      const int j = tid / kHeads, h = tid % kHeads;
      float M = -INFINITY;
      for (int jj = 0; jj < nsp; ++jj) M = fmaxf(M, w_s[jj][h]);
      const float e = f_l[j][h] > 0.0f ? expf(w_s[j][h] - M) : 0.0f;
      e_s[j][h] = e;
      f_l[j][h] *= e;  // l_j e_j, read by every j below
      if (j == 0) M_s[h] = M;
    }
    __syncthreads();
    if (tid < nsp * kHeads) {
      const int j = tid / kHeads, h = tid % kHeads;
      float Lsum = 0.0f;
      for (int jj = 0; jj < nsp; ++jj) Lsum += f_l[jj][h];   // fixed order
      w_s[j][h] = Lsum > 0.0f ? e_s[j][h] / Lsum : 0.0f;
      if (j == 0 && rank == 0 && a.lse) a.lse[(int64_t)qi * kHeads + h] = Lsum > 0.0f ? M_s[h] + logf(Lsum) : -INFINITY;
    }
    __syncthreads();
    for (int i0 = tid; i0 < n_items; i0 += 2 * kThreads) {
      if (i0 != tid) load_items(i0);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int i = i0 + u * kThreads;
        if (i >= n_items) break;
        const int h = h0 + i / (kHeadDim / 4), c4 = (i % (kHeadDim / 4)) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < kMaxClusterChunks; ++j) {   // fixed rank order
          if (j >= nsp) break;
          const float f = w_s[j][h];
          acc.x = fmaf(v[u][j].x, f, acc.x);
          acc.y = fmaf(v[u][j].y, f, acc.y);
          acc.z = fmaf(v[u][j].z, f, acc.z);
          acc.w = fmaf(v[u][j].w, f, acc.w);
        }
        const int64_t o = ((int64_t)qi * kHeads + h) * kHeadDim + c4;
        if (a.out_f32) *reinterpret_cast<float4*>(a.out_f32 + o) = acc;
        const __nv_bfloat162 b0 = __floats2bfloat162_rn(acc.x, acc.y), b1 = __floats2bfloat162_rn(acc.z, acc.w);
        *reinterpret_cast<uint2*>(a.out + o) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1));
      }
    }
    cl.sync();  // the other ranks have finished reading this CTA's shared memory
  } else {
    // ---- partial O = O_hi + O_lo (unnormalised, fp32) and (max, sum) to the workspace ----
    float* po = a.part_o + ((int64_t)lq * a.n_split + split) * kHeads * kHeadDim;
    if (ok) {
#pragma unroll
      for (int hh = 0; hh < kHeads; hh += 32) {
        uint32_t rh[32], rl[32];
        tc::tmem_ld_32x32b_x32(o_base + (uint32_t)hh, rh);
        tc::tmem_ld_32x32b_x32(o_base + (uint32_t)(kHeads + hh), rl);
        tc::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          po[(hh + j) * kHeadDim + c_own] = __uint_as_float(rh[j]) + __uint_as_float(rl[j]);
      }
    }
    if (tid < kHeads) {
      float* ml = a.part_ml + (((int64_t)lq * a.n_split + split) * kHeads + tid) * 2;
      ml[0] = m_s[tid];
      ml[1] = ok ? l_s[tid] : 0.0f;
    }
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
