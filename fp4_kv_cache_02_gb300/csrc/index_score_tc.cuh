// index_score_tc.cuh -- tensor-core lightning-indexer scan (included by
// index_score.cu, which owns the error word g_index_error).
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" section
// 2.3 / 2.4.4 and mer.dev notes section 4.4: every visible entry is scored as
// s = sum_h w_h ReLU(q_h . k) with 32 heads x 128 channels, q and k both
// MXFP4 (E2M1 values, one E8M0 scale per 32).
//
// One CTA scans 128-key tiles of one sequence: a contiguous run, or (claimed
// mode, dense rows) a fixed first range of one pipeline depth and then tiles
// claimed two at a time from the sequence's counter, so that CTAs with a
// larger share of the memory bandwidth take more of them:
//   warp 4       TMA producer: 128 x 64 B E2M1 tile (3-D tensor map, 64-byte
//                swizzle) + the tile's 512 B of E8M0 scales (bulk copy) per
//                pipeline stage;
//   warp 5       MMA issuer: rearranges the tile's scales for tcgen05.cp into
//                tensor memory, then issues two block-scaled MXF4 MMAs
//                (M = 128 keys, N = 32 heads, K = 64 each) into one of two
//                tensor-memory accumulators;
//   warps 0..3   epilogue: tcgen05.ld of each key's 32 head dots, ReLU, the
//                w-weighted fp32 sum, masking past n_visible, coalesced store.
// The scan is HBM-bound at 68 bytes per key; the tensor cores do the 4,096
// multiply-adds per key that CUDA cores could not sustain at that rate.
#pragma once

#include <cudaTypedefs.h>

#include "codec_blocks.cuh"
#include "tc_common.cuh"

namespace csa2 {
namespace scan_tc {

constexpr int kStages = 6;
constexpr int kTileRows = 128;
constexpr int kTileBytes = kTileRows * kIkBytes;    // 8192
constexpr int kSfBytes = kTileRows * kIkScales;     // 512
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 128;
__host__ __device__ constexpr uint32_t acc_col(int a) { return 32u * (uint32_t)a; }      // 2 x 32 fp32 columns
__host__ __device__ constexpr uint32_t sfa_col(int a) { return 64u + 8u * (uint32_t)a; }  // 2 x 4 scale columns
constexpr uint32_t kSfbCol = 80;

// shared-memory layout (offsets from a 1024-byte-aligned base)
constexpr int kOffA = 0;
constexpr int kOffSfRaw = kOffA + kStages * kTileBytes;
constexpr int kOffSfT = kOffSfRaw + kStages * kSfBytes;
constexpr int kOffQ = kOffSfT + kStages * kSfBytes;   // 1024-aligned: kStages * 9216 is
constexpr int kOffSfb = kOffQ + kIdxHeads * kIkBytes; // 2048 bytes of q
constexpr int kOffBars = kOffSfb + 512;
constexpr int kNumBars = 2 * kStages + 4;
constexpr int kOffMisc = kOffBars + kNumBars * 8;
constexpr int kOffHist = kOffMisc + 16;               // Top-K histogram of this CTA's scores
constexpr int kRing = 16;                             // tile index of each tile in flight (claimed mode)
constexpr int kOffRing = kOffHist + kTopkHistBins * 4;
constexpr int kSmemBytes = kOffRing + kRing * 4 + 1024;  // + alignment slack
static_assert(kOffQ % 1024 == 0, "q operand must be 1024-byte aligned");

struct Params {
  const uint8_t* ik_data;  // read directly (cp.async) in the positions mode
  const int32_t* positions;  // optional [B][n_pos] cache positions; NULL = 0..n_pos-1
  const uint8_t* q_data;
  const uint8_t* q_e8m0;
  const float* w;
  const uint8_t* ik_scale;
  int64_t cap;
  const int32_t* n_visible;
  int64_t n_pos;
  float* scores;
  int32_t tiles_per_cta;
  uint32_t* hist;  // optional [B][kTopkHistBins] Top-K histogram (zeroed by the caller)
  float* bmax;     // optional [B][ceil(n_pos / 8)] block maxima for the candidate pool (dense mode)
  // 1 when the preceding kernel in the stream writes only the workspace (the
  // histogram clear): then the cache, q and positions are read at once and
  // only the epilogue's writes wait for that kernel
  int32_t early_reads;
  // optional [B][32][128] bf16 indexer q: quantised to MXFP4 in the prologue
  // (the same block encoder as csa2_quant_mxfp4) instead of reading q_data
  const uint16_t* q_bf16;
  // optional tile counters, sequence b's at tile_ctr[b * tile_ctr_stride],
  // zero when the preceding kernel ends (dense mode): after its first
  // `claim0` tiles (a fixed range, read at once) each CTA of a sequence claims
  // `claim` tiles at a time from the counter, so that CTAs with a larger share
  // of the memory bandwidth take more tiles
  int32_t* tile_ctr;
  int32_t tile_ctr_stride;
  int32_t claim0;
  int32_t claim;
  // optional, beside tile_ctr (same stride): CTAs of the sequence that have
  // finished; the last one puts both words back to zero for the next launch
  int32_t* tile_done;
};

__global__ void __launch_bounds__(kThreads, 3)
    index_score_tc_kernel(const __grid_constant__ CUtensorMap tmap_ik, Params p) {
  if (p.early_reads)
    pdl_launch_dependents();
  else
    pdl_begin();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = tc::smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  uint8_t* sA = sm + kOffA;
  uint8_t* sSfRaw = sm + kOffSfRaw;
  uint8_t* sSfT = sm + kOffSfT;
  uint8_t* sQ = sm + kOffQ;
  uint8_t* sSfb = sm + kOffSfb;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kOffBars);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + kOffMisc + 4);
  uint32_t* s_hist = reinterpret_cast<uint32_t*>(sm + kOffHist);
  volatile int32_t* s_ring = reinterpret_cast<volatile int32_t*>(sm + kOffRing);
  const bool with_hist = p.hist != nullptr;
  const bool pos_mode = p.positions != nullptr;
  // claimed mode: tiles come from the sequence's counter, their indices pass
  // from the producer to the MMA warp and the epilogue through s_ring; a tile
  // index of -1 ends the stream
  const bool claimed = !pos_mode && p.tile_ctr != nullptr;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // grid (sequences, chunks): consecutive CTAs belong to different sequences,
  // so each sequence's CTAs spread over the SMs of both dies
  const int b = blockIdx.x;
  const int chunk = blockIdx.y, n_chunks = gridDim.y;
  const int64_t n_tiles_all = (p.n_pos + kTileRows - 1) / kTileRows;
  int64_t nv = (int64_t)p.n_visible[b];
  // positions mode: a listed position is scored when it is below n_visible
  // (and the capacity); dense mode: entries 0..nv-1 of the list
  const int64_t nv_pos = nv < 0 ? 0 : (nv > p.cap ? p.cap : nv);
  nv = nv < 0 ? 0 : (nv > p.n_pos ? p.n_pos : nv);
  const int64_t t_begin = (int64_t)chunk * p.tiles_per_cta;
  int64_t t_end_all = t_begin + p.tiles_per_cta;
  if (t_end_all > n_tiles_all) t_end_all = n_tiles_all;
  int64_t t_end = pos_mode ? t_end_all : (nv + kTileRows - 1) / kTileRows;
  if (t_end > t_end_all) t_end = t_end_all;
  const int n_tiles = t_end > t_begin ? (int)(t_end - t_begin) : 0;
  // claimed mode: tiles 0 .. t_vis-1 of the sequence hold visible entries
  const int64_t t_vis_ = (nv + kTileRows - 1) / kTileRows;
  const int32_t t_vis = (int32_t)(t_vis_ < n_tiles_all ? t_vis_ : n_tiles_all);

  // ---- set-up: barriers, the q operand (B) and its scales, tensor memory ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], pos_mode ? 32 : 1);  // positions mode: one cp.async arrival per producer lane
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&acc_full[a], 1);
      tc::mbar_init(&acc_empty[a], 4);  // one arrival per epilogue warp
    }
    *s_abort = 0;
    tc::fence_mbar_init();
  }
  if (threadIdx.x < 128 && p.q_bf16) {
    // q: head r, channels 32c .. 32c+31 -> one MXFP4 block: 16 bytes at its
    // SW64 place and the E8M0 byte, the four bytes of a head gathered by shuffles
    const int r = threadIdx.x >> 2, c = threadIdx.x & 3;
    const uint4* src = reinterpret_cast<const uint4*>(p.q_bf16 + ((int64_t)b * kIdxHeads + r) * kIdxDim + c * 32);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = src[i];
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
    uint4 d;
    uint8_t e;
    encode_mxfp4_block(w, d, e);
    *reinterpret_cast<uint4*>(sQ + tc::sw64_offset(r, c)) = d;
    uint32_t sb = (uint32_t)e << (8 * c);
    sb |= __shfl_xor_sync(0xffffffffu, sb, 1);
    sb |= __shfl_xor_sync(0xffffffffu, sb, 2);
    if (c == 0) *reinterpret_cast<uint4*>(sSfb + r * 16) = make_uint4(sb, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
  } else if (threadIdx.x < 128) {
    // q: 32 rows x 64 B, K-major with the 64-byte swizzle
    const int r = threadIdx.x >> 2, c = threadIdx.x & 3;
    uint4 v = *reinterpret_cast<const uint4*>(p.q_data + ((int64_t)b * kIdxHeads + r) * kIkBytes + c * 16);
    *reinterpret_cast<uint4*>(sQ + tc::sw64_offset(r, c)) = v;
  } else if (threadIdx.x < 160 && !p.q_bf16) {
    // scales of q for tcgen05.cp: row i holds the four E8M0 bytes of head i
    // (bytes for rows i+32, i+64, i+96 do not exist for N = 32 and are 2^0)
    const int i = threadIdx.x - 128;
    uint32_t s = *reinterpret_cast<const uint32_t*>(p.q_e8m0 + ((int64_t)b * kIdxHeads + i) * kIkScales);
    *reinterpret_cast<uint4*>(sSfb + i * 16) = make_uint4(s, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
  }
  if (with_hist)
    for (int i = threadIdx.x; i < kTopkHistBins; i += kThreads) s_hist[i] = 0u;
  tc::fence_proxy_async_smem();
  if (warp == kMmaWarp) tc::tmem_alloc(s_tmem, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == kProducerWarp && pos_mode) {
    // ---- gather producer: lane l copies rows 4l..4l+3 of each tile (64 data
    // bytes in four 16-byte chunks at their SW64 places, 4 scale bytes);
    // rows whose position is not visible are zero-filled ----
    const int32_t* plist = p.positions + (int64_t)b * p.n_pos;
    int32_t pv[4];
    const auto fetch = [&](int i) {
      const int64_t base = (t_begin + i) * kTileRows + lane * 4;
#pragma unroll
      for (int q = 0; q < 4; ++q) pv[q] = base + q < p.n_pos ? plist[base + q] : -1;
    };
    if (n_tiles > 0) fetch(0);
    int i = 0;
    for (; i < n_tiles; ++i) {
      const int s = i % kStages;
      const uint32_t ph = (uint32_t)(i / kStages) & 1u;
      const bool ok = tc::mbar_wait_bounded(&empty[s], ph ^ 1u, s_abort, &g_index_error);
      if (!__all_sync(0xffffffffu, ok)) break;
      int32_t cur[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) cur[q] = pv[q];
      if (i + 1 < n_tiles) fetch(i + 1);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t r = (uint32_t)(lane * 4 + q);
        const bool valid = cur[q] >= 0 && cur[q] < nv_pos;
        const int64_t src = (int64_t)b * p.cap + (valid ? cur[q] : 0);
        const uint32_t nb = valid ? 16u : 0u;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tc::cp_async_16(sA + s * kTileBytes + tc::sw64_offset(r, (uint32_t)c), p.ik_data + src * kIkBytes + c * 16,
                          nb);
        tc::cp_async_4(sSfRaw + s * kSfBytes + r * 4, p.ik_scale + src * kIkScales, valid ? 4u : 0u);
      }
      tc::cp_async_mbar_arrive(&full[s]);
    }
    tc::cp_async_wait_all();  // nothing of this lane is in flight when the CTA ends
    __syncwarp();
  } else if (warp == kProducerWarp) {
    // ---- TMA producer ----
    if (lane == 0) {
      int issued = 0;
      const auto issue = [&](int i, int64_t tile) -> bool {
        const int s = i % kStages;
        const uint32_t ph = (uint32_t)(i / kStages) & 1u;
        if (!tc::mbar_wait_bounded(&empty[s], ph ^ 1u, s_abort, &g_index_error)) return false;
        const int64_t row0 = tile * kTileRows;
        if (claimed) s_ring[i % kRing] = (int32_t)tile;
        tc::mbar_arrive_expect_tx(&full[s], kTileBytes + kSfBytes);
        tc::tma_load_3d(sA + s * kTileBytes, &tmap_ik, 0, (int32_t)row0, b, &full[s]);
        tc::bulk_load(sSfRaw + s * kSfBytes, p.ik_scale + ((int64_t)b * p.cap + row0) * kIkScales, kSfBytes,
                      &full[s]);
        return true;
      };
      if (claimed) {
        bool ok = true;
        // the fixed first range: tiles [x * claim0, x * claim0 + claim0)
        const int32_t c0 = (int32_t)chunk * p.claim0;
        for (int32_t t = c0; ok && t < c0 + p.claim0 && t < t_vis; ++t) {
          ok = issue(issued, t);
          if (ok) ++issued;
        }
        // the counter is cleared by the preceding kernel
        if (p.early_reads) pdl_wait();
        const int32_t base = (int32_t)n_chunks * p.claim0;
        const int32_t step = p.claim > 0 ? p.claim : 1;
        while (ok && base < t_vis) {
          const int32_t c = base + atomicAdd(p.tile_ctr + (int64_t)b * p.tile_ctr_stride, step);
          if (c >= t_vis) break;
          const int32_t ce = c + step < t_vis ? c + step : t_vis;
          for (int32_t t = c; ok && t < ce; ++t) {
            ok = issue(issued, t);
            if (ok) ++issued;
          }
        }
        if (ok) {
          // the end of the stream: one more stage, no bytes, tile index -1
          const int s = issued % kStages;
          if (tc::mbar_wait_bounded(&empty[s], ((uint32_t)(issued / kStages) & 1u) ^ 1u, s_abort, &g_index_error)) {
            s_ring[issued % kRing] = -1;
            tc::mbar_arrive(&full[s]);
          }
        }
      } else {
        for (int i = 0; i < n_tiles; ++i) {
          if (!issue(i, t_begin + i)) break;
          ++issued;
        }
      }
      if (*s_abort) {
        // let copies already in flight land before the CTA's memory goes away
        for (int i = issued - kStages; i < issued; ++i)
          if (i >= 0) tc::mbar_wait_bounded(&full[i % kStages], (uint32_t)(i / kStages) & 1u, s_abort,
                                            &g_index_error, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer ----
    const uint32_t q_addr = tc::smem_u32(sQ);
    const uint64_t bdesc0 = tc::smem_desc(q_addr, 0, 512, tc::kSwizzle64B);
    const uint64_t bdesc1 = tc::smem_desc(q_addr + 32, 0, 512, tc::kSwizzle64B);
    constexpr uint32_t idesc0 = tc::idesc_mxf4(128, 32, 0, 0);
    constexpr uint32_t idesc1 = tc::idesc_mxf4(128, 32, 2, 2);
    // q's scales into tensor memory, for every CTA that may score a tile (in
    // claimed mode any CTA of the sequence may)
    if (lane == 0 && (claimed || n_tiles > 0))
      tc::tmem_cp_32x128_x4(tmem + kSfbCol, tc::smem_desc(tc::smem_u32(sSfb), 0, 128, tc::kSwizzleNone));
    __syncwarp();
    int last = -1;
    for (int i = 0; claimed || i < n_tiles; ++i) {
      const int s = i % kStages;
      const uint32_t ph = (uint32_t)(i / kStages) & 1u;
      const int a = i & 1;
      const uint32_t aph = (uint32_t)(i >> 1) & 1u;
      bool ok = tc::mbar_wait_bounded(&acc_empty[a], aph ^ 1u, s_abort, &g_index_error) &&
                tc::mbar_wait_bounded(&full[s], ph, s_abort, &g_index_error);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (claimed && s_ring[i % kRing] < 0) {
        if (lane == 0) tc::mbar_arrive(&acc_full[a]);  // passes the end on to the epilogue
        break;
      }
      // scales of keys lane, lane+32, lane+64, lane+96 -> one 16-byte row
      const uint32_t* raw = reinterpret_cast<const uint32_t*>(sSfRaw + s * kSfBytes);
      uint4 v = make_uint4(raw[lane], raw[lane + 32], raw[lane + 64], raw[lane + 96]);
      *reinterpret_cast<uint4*>(sSfT + s * kSfBytes + lane * 16) = v;
      tc::fence_proxy_async_smem();
      __syncwarp();
      tc::tc_fence_after();
      if (lane == 0) {
        const uint32_t sfa = tmem + sfa_col(a);
        const uint32_t d = tmem + acc_col(a);
        tc::tmem_cp_32x128_x4(sfa, tc::smem_desc(tc::smem_u32(sSfT + s * kSfBytes), 0, 128, tc::kSwizzleNone));
        const uint32_t a_addr = tc::smem_u32(sA + s * kTileBytes);
        tc::mma_mxf4(d, tc::smem_desc(a_addr, 0, 512, tc::kSwizzle64B), bdesc0, idesc0, sfa, tmem + kSfbCol, 0);
        tc::mma_mxf4(d, tc::smem_desc(a_addr + 32, 0, 512, tc::kSwizzle64B), bdesc1, idesc1, sfa,
                     tmem + kSfbCol, 1);
        tc::mma_commit(&empty[s]);
        tc::mma_commit(&acc_full[a]);
      }
      last = i;
      __syncwarp();
    }
    if (*s_abort && last >= 0 && lane == 0)  // MMAs must finish before tensor memory is freed
      tc::mbar_wait_bounded(&acc_full[last & 1], (uint32_t)(last >> 1) & 1u, s_abort, &g_index_error,
                            100000000ull);
    __syncwarp();
  } else {
    // ---- epilogue: warps 0..3, one key row per thread ----
    if (p.early_reads) pdl_wait();  // the scores, maxima and histogram are written below
    float wr[kIdxHeads];
#pragma unroll
    for (int h = 0; h < kIdxHeads; ++h) wr[h] = p.w[(int64_t)b * kIdxHeads + h];
    const int row = warp * 32 + lane;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float* out = p.scores + (int64_t)b * p.n_pos;
    for (int i = 0; claimed || i < n_tiles; ++i) {
      const int a = i & 1;
      const uint32_t aph = (uint32_t)(i >> 1) & 1u;
      // warp-uniform outcome: tcgen05.ld below needs the whole warp
      if (!__all_sync(0xffffffffu, tc::mbar_wait_bounded(&acc_full[a], aph, s_abort, &g_index_error))) break;
      const int64_t tile = claimed ? (int64_t)s_ring[i % kRing] : t_begin + i;
      if (tile < 0) break;
      tc::tc_fence_after();
      uint32_t r[32];
      tc::tmem_ld_32x32b_x32(tmem + lane_base + acc_col(a), r);
      tc::tmem_ld_wait();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty[a]);
      float sc = 0.0f;
#pragma unroll
      for (int h = 0; h < kIdxHeads; ++h) sc = fmaf(wr[h], fmaxf(__uint_as_float(r[h]), 0.0f), sc);
      const int64_t li = tile * kTileRows + row;  // list index
      bool valid = li < nv;
      if (pos_mode) {
        const int32_t pp = li < p.n_pos ? p.positions[(int64_t)b * p.n_pos + li] : -1;
        valid = pp >= 0 && pp < nv_pos;
      }
      if (li < p.n_pos) out[li] = valid ? sc : -INFINITY;
      if (p.bmax) {
        // maximum over the block of 8 consecutive entries (8 consecutive lanes);
        // entries past n_visible and NaN scores take no part
        float v = valid && !isnan(sc) ? sc : -INFINITY;
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
        if ((lane & 7) == 0 && li < p.n_pos) p.bmax[(int64_t)b * ((p.n_pos + 7) / 8) + li / 8] = v;
      }
      if (with_hist && valid && score_is_candidate(sc))
        atomicAdd(&s_hist[score_key(sc) >> (32 - kTopkHistBits)], 1u);
    }
    // tiles past the visible entries: this CTA's range, or in claimed mode
    // every n_chunks-th tile from t_vis + chunk
    const int64_t fill_lo = claimed ? t_vis + (int64_t)chunk : (t_begin > t_end ? t_begin : t_end);
    const int64_t fill_hi = claimed ? n_tiles_all : t_end_all;
    const int64_t fill_step = claimed ? (int64_t)n_chunks : 1;
    for (int64_t t = fill_lo; t < fill_hi; t += fill_step) {
      const int64_t lo = t * kTileRows;
      const int64_t hi = lo + kTileRows < p.n_pos ? lo + kTileRows : p.n_pos;
      for (int64_t pos = lo + threadIdx.x; pos < hi; pos += 128) out[pos] = -INFINITY;
      if (p.bmax) {
        float* bm = p.bmax + (int64_t)b * ((p.n_pos + 7) / 8);
        for (int64_t j = lo / 8 + threadIdx.x; j < (hi + 7) / 8; j += 128) bm[j] = -INFINITY;
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  if (claimed && p.tile_done && threadIdx.x == 0) {
    // every CTA of the sequence has made its last claim once all have arrived here
    __threadfence();
    int32_t* done = p.tile_done + (int64_t)b * p.tile_ctr_stride;
    if (atomicAdd(done, 1) == n_chunks - 1) {
      p.tile_ctr[(int64_t)b * p.tile_ctr_stride] = 0;
      *done = 0;
    }
  }
  if (with_hist) {
    if (p.early_reads) pdl_wait();
    uint32_t* gh = p.hist + (int64_t)b * kTopkHistBins;
    for (int i = threadIdx.x; i < kTopkHistBins; i += kThreads)
      if (s_hist[i]) atomicAdd(&gh[i], s_hist[i]);
  }
}

}  // namespace scan_tc
}  // namespace csa2
