// prefill_score_tc.cuh -- tensor-core indexer scores for a prefill chunk.
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", section
// 2.3 (indexer scores with MXFP4 q and k) and the mer.dev notes on the
// prefill indexer (its cost grows with the square of the context): T queries
// at positions p0 .. p0+T-1 of one sequence each score every entry at or
// before their own position,
//
//   s[t][j] = sum_h w[t][h] * ReLU( qhat[t][h] . khat[j] ),  j <= p0 + t,
//
// and -inf for later entries.
//
// One CTA keeps a block of 32 queries (32 x 32 = 1024 MXFP4 rows of q, the
// B operand) in shared memory and streams a chunk of 128-entry key tiles (the
// A operand) through a TMA pipeline. Per key tile the MMA warp issues eight
// 128 x 128 x 128 block-scaled MXF4 products, one per group of four queries,
// into three TMEM accumulators in rotation. Sixteen epilogue warps in four
// sets take the groups in turn: warp w of a set reads TMEM lanes 32(w % 4)..
// (32 keys) and the 4 x 32 head columns of the group, two queries at a time,
// frees the accumulator after the second load, applies ReLU (half of the
// heads by max, half as x + |x| = 2 ReLU(x), to share the ALU and FMA pipes),
// weights the heads with packed f32x2 FMAs and stores 32 consecutive scores of
// each query. The epilogue's issue rate, not the tensor pipe, bounds this
// kernel: about three instructions per (entry, head) value against 128 MACs
// of tensor work, so the per-group costs (barrier wait, loads, release, mask
// and address arithmetic) are taken once per four queries, and the causal
// mask and bounds only on tiles that some query of the block does not see
// whole.
#pragma once

#include <cuda.h>

#include "tc_common.cuh"

namespace csa2 {
namespace prefill_tc {

constexpr int kQBlock = 32;                   // queries per CTA
constexpr int kGroupQ = 4;                    // queries per MMA (N = 4 x 32 heads)
constexpr int kGroups = kQBlock / kGroupQ;    // 8
constexpr int kN = kGroupQ * kIdxHeads;       // 128
constexpr int kTileRows = 128;                // keys per tile (M)
constexpr int kStages = 4;
constexpr int kChunkTiles = 64;               // key tiles per CTA
constexpr int kTileBytes = kTileRows * kIkBytes;  // 8192
constexpr int kSfBytes = kTileRows * kIkScales;   // 512
constexpr int kQRows = kQBlock * kIdxHeads;       // 1024
constexpr int kAcc = 3;                           // TMEM accumulators in rotation
constexpr int kSets = 4;                          // epilogue warp sets, taking groups in rotation
constexpr int kSetWarps = 4;                      // warps of a set: one per lane quadrant
constexpr int kEpiWarps = kSets * kSetWarps;      // 16
constexpr int kProducerWarp = kEpiWarps;          // 16
constexpr int kMmaWarp = kEpiWarps + 1;           // 17
constexpr int kThreads = (kEpiWarps + 2) * 32;    // 576
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t acc_col(int a) { return 128u * (uint32_t)a; }      // 3 x 128 fp32 columns
__host__ __device__ constexpr uint32_t sfa_col(int a) { return 384u + 4u * (uint32_t)a; }  // 2 x 4 scale columns
constexpr uint32_t kSfbCol = 392;                                                          // 8 groups x 4 columns

// shared-memory layout (offsets from a 1024-byte-aligned base)
constexpr int kOffQ = 0;                                  // 1024 rows x 64 B, SW64 K-major
constexpr int kOffA = kOffQ + kQRows * kIkBytes;          // 65536
constexpr int kOffSfT = kOffA + kStages * kTileBytes;        // key scales, transposed for tcgen05.cp
constexpr int kOffSfb = kOffSfT + kStages * kSfBytes;     // 8 groups x 512 B, transposed for tcgen05.cp
constexpr int kOffW = kOffSfb + kGroups * 512;            // [32 queries][32 heads] fp32
constexpr int kOffBars = kOffW + kQBlock * kIdxHeads * 4;
constexpr int kNumBars = 2 * kStages + kSets + kAcc;
constexpr int kOffMisc = kOffBars + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;          // + alignment slack
static_assert(kOffA % 1024 == 0 && kOffSfb % 16 == 0, "operand alignment");
static_assert(kGroups % kSets == 0, "a tile's groups divide evenly over the epilogue sets");
static_assert(kSets >= kAcc, "a set barrier runs at most one phase ahead of its set");

struct Params {
  const uint8_t* q_e8m0;   // [T][32][4]
  const float* w;          // [T][32]
  const uint8_t* ik_scale; // [n_entries][4]
  int64_t n_entries;
  int64_t p0;              // token position of query 0
  int32_t T;
  int32_t m;               // tokens per entry: query t sees entries j < (p0 + t + 1) / m
  float* scores;           // [T][n_entries]
};

__device__ __forceinline__ unsigned long long pack_f32x2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ unsigned long long pack_u32x2(uint32_t lo, uint32_t hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ float sum_f32x2(unsigned long long v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo + hi;
}
// acc += a * b on two fp32 lanes
__device__ __forceinline__ void fma_f32x2(unsigned long long& acc, unsigned long long a, unsigned long long b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

// grid (key chunks, query blocks)
__global__ void __launch_bounds__(kThreads, 1)
    prefill_score_tc_kernel(const __grid_constant__ CUtensorMap tmap_ik, const __grid_constant__ CUtensorMap tmap_q,
                            Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = tc::smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  uint8_t* sQ = sm + kOffQ;
  uint8_t* sA = sm + kOffA;
  uint8_t* sSfT = sm + kOffSfT;
  uint8_t* sSfb = sm + kOffSfb;
  float* sW = reinterpret_cast<float*>(sm + kOffW);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kOffBars);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;   // per epilogue set: its next group is in TMEM
  uint64_t* acc_empty = acc_full + kSets; // per accumulator: drained into registers
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + kOffMisc + 4);
  uint64_t* qbar = reinterpret_cast<uint64_t*>(sm + kOffMisc + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.y * kQBlock;
  const int64_t tiles_all = (p.n_entries + kTileRows - 1) / kTileRows;
  // entries visible to the block's last query, in tiles
  const int64_t last_t = min((int64_t)t0 + kQBlock, (int64_t)p.T) - 1;
  const int64_t last_vis = (p.p0 + last_t + 1) / p.m;        // entries the last query sees
  int64_t vis_tiles = (last_vis + kTileRows - 1) / kTileRows;
  if (vis_tiles > tiles_all) vis_tiles = tiles_all;
  const int64_t c0 = (int64_t)blockIdx.x * kChunkTiles;
  const int64_t c1 = min(c0 + kChunkTiles, tiles_all);
  const int64_t m1 = min(c1, vis_tiles);                  // tiles [c0, m1) need the MMA
  const int n_mma_tiles = m1 > c0 ? (int)(m1 - c0) : 0;

  // ---- set-up ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1 + 32);  // producer lane 0 (TMA bytes) + the 32 lanes' scale rows
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < kAcc; ++a) {
      tc::mbar_init(&acc_empty[a], kSetWarps);  // one arrival per warp of the set
    }
    // a set's groups are committed in its own order, at most one ahead of the
    // set (the MMA after that needs an accumulator the set still holds), so
    // one parity bit per set barrier tells its phases apart; a barrier shared by
    // the sets would not
    for (int k = 0; k < kSets; ++k) tc::mbar_init(&acc_full[k], 1);
    tc::mbar_init(qbar, 1);
    *s_abort = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && n_mma_tiles > 0) {
    // the block's q rows (OOB rows past T read as zero)
    tc::mbar_arrive_expect_tx(qbar, kQRows * kIkBytes);
    for (int i = 0; i < kQRows / 256; ++i)
      tc::tma_load_2d(sQ + i * 256 * kIkBytes, &tmap_q, 0, t0 * kIdxHeads + i * 256, qbar);
  }
  if (threadIdx.x < kGroups * 32) {
    // q scales, transposed for tcgen05.cp: group g, lane l -> rows l, l+32, l+64, l+96 of the group
    const int g = threadIdx.x >> 5, l = threadIdx.x & 31;
    uint32_t v[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int row = g * kN + l + 32 * c;  // row = query-in-block * 32 + head
      const int t = t0 + row / kIdxHeads;
      v[c] = t < p.T ? *reinterpret_cast<const uint32_t*>(p.q_e8m0 + ((int64_t)t * kIdxHeads + row % kIdxHeads) *
                                                                         kIkScales)
                     : 0x7F7F7F7Fu;
    }
    *reinterpret_cast<uint4*>(sSfb + g * 512 + l * 16) = make_uint4(v[0], v[1], v[2], v[3]);
  }
  for (int i = threadIdx.x; i < kQBlock * kIdxHeads; i += kThreads) {
    const int t = t0 + i / kIdxHeads;
    sW[i] = t < p.T ? p.w[(int64_t)t * kIdxHeads + i % kIdxHeads] : 0.0f;
  }
  tc::fence_proxy_async_smem();
  if (warp == kMmaWarp) tc::tmem_alloc(s_tmem, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == kProducerWarp) {
    // ---- producer: key tile by TMA (lane 0); the tile's 128 scale words by
    // plain loads, lane l writing the 16-byte tcgen05.cp row of keys l, l+32,
    // l+64, l+96 (the next tile's words are loaded while this one is placed) ----
    uint32_t sv[4];
    const auto fetch = [&](int i) {
      const int64_t row0 = (c0 + i) * kTileRows;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t r = row0 + lane + 32 * q;
        sv[q] = r < p.n_entries ? __ldg(reinterpret_cast<const unsigned int*>(p.ik_scale + r * kIkScales))
                                : 0x7F7F7F7Fu;
      }
    };
    if (n_mma_tiles > 0) fetch(0);
    int i = 0;
    for (; i < n_mma_tiles; ++i) {
      const int s = i % kStages;
      const uint32_t ph = (uint32_t)(i / kStages) & 1u;
      const bool ok = tc::mbar_wait_bounded(&empty[s], ph ^ 1u, s_abort, &g_index_error);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (lane == 0) {
        tc::mbar_arrive_expect_tx(&full[s], kTileBytes);
        tc::tma_load_2d(sA + s * kTileBytes, &tmap_ik, 0, (int32_t)((c0 + i) * kTileRows), &full[s]);
      }
      *reinterpret_cast<uint4*>(sSfT + s * kSfBytes + lane * 16) = make_uint4(sv[0], sv[1], sv[2], sv[3]);
      tc::fence_proxy_async_smem();  // the scale row is read by tcgen05.cp (async proxy)
      tc::mbar_arrive(&full[s]);
      if (i + 1 < n_mma_tiles) fetch(i + 1);
    }
    if (*s_abort && lane == 0) {
      // TMA tiles already in flight must land before the CTA's memory goes away
      for (int j = i - kStages; j < i; ++j)
        if (j >= 0) tc::mbar_wait_bounded(&full[j % kStages], (uint32_t)(j / kStages) & 1u, s_abort, &g_index_error,
                                          100000000ull);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer: one lane; descriptors advance by constant offsets ----
    if (lane == 0) {
      bool ok = n_mma_tiles == 0 || tc::mbar_wait_bounded(qbar, 0, s_abort, &g_index_error);
      if (ok && n_mma_tiles > 0) {
        tc::tc_fence_after();
        for (int g = 0; g < kGroups; ++g)
          tc::tmem_cp_32x128_x4(tmem + kSfbCol + 4u * g,
                                tc::smem_desc(tc::smem_u32(sSfb + g * 512), 0, 128, tc::kSwizzleNone));
      }
      constexpr uint32_t idesc0 = tc::idesc_mxf4(kTileRows, kN, 0, 0);
      constexpr uint32_t idesc1 = tc::idesc_mxf4(kTileRows, kN, 2, 2);
      // descriptor address fields count 16-byte units
      const uint64_t a_desc0 = tc::smem_desc(tc::smem_u32(sA), 0, 512, tc::kSwizzle64B);
      const uint64_t b_desc0 = tc::smem_desc(tc::smem_u32(sQ), 0, 512, tc::kSwizzle64B);
      const uint64_t sf_desc0 = tc::smem_desc(tc::smem_u32(sSfT), 0, 128, tc::kSwizzleNone);
      int a = 0;              // accumulator of the next group
      uint32_t uses = 0;      // bit a: parity of the uses of accumulator a so far
      int last_f = -1;        // set barrier of the last commit, and its parity
      uint32_t last_par = 0;
      for (int i = 0; ok && i < n_mma_tiles; ++i) {
        const int s = i % kStages;
        ok = tc::mbar_wait_bounded(&full[s], (uint32_t)(i / kStages) & 1u, s_abort, &g_index_error);
        if (!ok) break;
        tc::tc_fence_after();
        const uint32_t sfa = tmem + sfa_col(i & 1);
        tc::tmem_cp_32x128_x4(sfa, sf_desc0 + (uint64_t)((s * kSfBytes) >> 4));
        const uint64_t ad = a_desc0 + (uint64_t)((s * kTileBytes) >> 4);
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
          const uint32_t par = (uses >> a) & 1u;
          ok = tc::mbar_wait_bounded(&acc_empty[a], par ^ 1u, s_abort, &g_index_error);
          if (!ok) break;
          tc::tc_fence_after();
          const uint32_t d = tmem + acc_col(a);
          const uint64_t bd = b_desc0 + (uint64_t)((g * kN * kIkBytes) >> 4);
          const uint32_t sfb = tmem + kSfbCol + 4u * g;
          tc::mma_mxf4(d, ad, bd, idesc0, sfa, sfb, 0);
          tc::mma_mxf4(d, ad + 2, bd + 2, idesc1, sfa, sfb, 1);  // second K half: +32 bytes
          tc::mma_commit(&acc_full[g % kSets]);
          last_f = g % kSets;
          last_par = (uint32_t)(i * (kGroups / kSets) + g / kSets) & 1u;
          uses ^= 1u << a;
          a = a == kAcc - 1 ? 0 : a + 1;
        }
        if (ok) tc::mma_commit(&empty[s]);
      }
      if (*s_abort && last_f >= 0)  // MMAs must finish before tensor memory is freed
        tc::mbar_wait_bounded(&acc_full[last_f], last_par, s_abort, &g_index_error, 100000000ull);
    }
    __syncwarp();
  } else {
    // ---- epilogue: set k (4 warps) drains groups g = k, k + 4 of every tile;
    // warp w of a set reads TMEM lanes 32(w % 4).. (32 keys) ----
    const int set = warp / kSetWarps, quad = warp % kSetWarps;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int64_t N = p.n_entries;
    const bool all_q = t0 + kQBlock <= p.T;  // no query of the block past T
    bool live = true;
    for (int i = 0; live && i < n_mma_tiles; ++i) {
      // per tile: this thread's entry, its last token, and whether every query
      // of the block sees the whole tile (then no mask and no bounds per store)
      const int64_t jt = (c0 + i) * kTileRows;
      const int64_t j = jt + quad * 32 + lane;
      const int64_t jm_last = j * p.m + (p.m - 1);
      const bool whole = all_q && jt + kTileRows <= N && (jt + kTileRows) * p.m - 1 <= p.p0 + t0;
      float* dst = p.scores + ((int64_t)t0 + kGroupQ * set) * N + j;
#pragma unroll 1
      for (int g = set; g < kGroups; g += kSets, dst += kSets * kGroupQ * N) {
        const int a = (i * kGroups + g) % kAcc;  // the MMA fills accumulators in rotation
        // warp-uniform outcome: tcgen05.ld below needs the whole warp
        const uint32_t par = (uint32_t)(i * (kGroups / kSets) + g / kSets) & 1u;
        if (!__all_sync(0xffffffffu, tc::mbar_wait_bounded(&acc_full[set], par, s_abort, &g_index_error))) {
          live = false;
          break;
        }
        tc::tc_fence_after();
        float e[kGroupQ];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          // queries 2 half, 2 half + 1 of the group: 2 x 32 head columns
          uint32_t r[2][32];
          tc::tmem_ld_32x32b_x32(tmem + acc_col(a) + lane_off + 64u * half, r[0]);
          tc::tmem_ld_32x32b_x32(tmem + acc_col(a) + lane_off + 64u * half + 32u, r[1]);
          tc::tmem_ld_wait();
          if (half == 1) {  // the accumulator is free once its last columns are in registers
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&acc_empty[a]);
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            uint32_t* x = r[k];
            // ReLU in place, so that head pairs stay in the register pairs the
            // tensor-memory load wrote (packed FMAs take them as they are):
            // heads 4m, 4m+1 by max (ALU pipe), heads 4m+2, 4m+3 as x + |x| =
            // 2 ReLU(x) (FMA pipe), halved at the end (exact)
#pragma unroll
            for (int h = 0; h < kIdxHeads; h += 4) {
              x[h] = __float_as_uint(fmaxf(__uint_as_float(x[h]), 0.0f));
              x[h + 1] = __float_as_uint(fmaxf(__uint_as_float(x[h + 1]), 0.0f));
              x[h + 2] = __float_as_uint(__uint_as_float(x[h + 2]) + fabsf(__uint_as_float(x[h + 2])));
              x[h + 3] = __float_as_uint(__uint_as_float(x[h + 3]) + fabsf(__uint_as_float(x[h + 3])));
            }
            const ulonglong2* wq = reinterpret_cast<const ulonglong2*>(sW + (g * kGroupQ + 2 * half + k) * kIdxHeads);
            unsigned long long am0 = 0ull, aa0 = 0ull, am1 = 0ull, aa1 = 0ull;
#pragma unroll
            for (int h = 0; h < kIdxHeads; h += 8) {
              const ulonglong2 wa = wq[h >> 2], wb = wq[(h >> 2) + 1];
              fma_f32x2(am0, pack_u32x2(x[h], x[h + 1]), wa.x);
              fma_f32x2(aa0, pack_u32x2(x[h + 2], x[h + 3]), wa.y);
              fma_f32x2(am1, pack_u32x2(x[h + 4], x[h + 5]), wb.x);
              fma_f32x2(aa1, pack_u32x2(x[h + 6], x[h + 7]), wb.y);
            }
            e[2 * half + k] = sum_f32x2(am0) + sum_f32x2(am1) + 0.5f * (sum_f32x2(aa0) + sum_f32x2(aa1));
          }
        }
        if (whole) {
          float* d = dst;
#pragma unroll
          for (int k = 0; k < kGroupQ; ++k, d += N) *d = e[k];
        } else {
          // entry j (tokens jm .. jm+m-1) is complete at the query's position p0 + t
#pragma unroll
          for (int k = 0; k < kGroupQ; ++k) {
            const int t = t0 + g * kGroupQ + k;
            if (t < p.T && j < N) dst[k * N] = jm_last <= p.p0 + t ? e[k] : -INFINITY;
          }
        }
      }
    }
    // tiles of the chunk past every query of the block
    const int64_t lo = max(m1, c0) * kTileRows;
    const int64_t hi = min(c1 * kTileRows, p.n_entries);
    const int et = threadIdx.x;  // 0 .. kEpiWarps * 32 - 1
    for (int qi = 0; qi < kQBlock && t0 + qi < p.T; ++qi)
      for (int64_t jj = lo + et; jj < hi; jj += kEpiWarps * 32) p.scores[(int64_t)(t0 + qi) * p.n_entries + jj] = -INFINITY;
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace prefill_tc
}  // namespace csa2
