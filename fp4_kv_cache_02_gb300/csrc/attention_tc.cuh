// attention_tc.cuh -- tensor-core sparse attention (included by attention.cu,
// which owns g_attn_error and AttnArgs).
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", section
// 2.3: each query attends to its selected main-KV entries together with the
// layer's SWA rows in one softmax; mer.dev notes section 1: 64 heads of dim
// 512 share the 512-channel latent as K and V.
//
// A query's rows are cut into tiles of 128: the SWA tiles first, then the
// tiles of selected entries. A thread-block cluster of C CTAs serves one
// query; CTA r takes the tiles whose index is r modulo C, and each tile gives
// one partial softmax (m, l, O) over its rows:
//   1. the SWA rows of a tile come by one bulk copy into a staging area; a
//      selected latent (256 B of codes + 32 B of scales) is loaded straight
//      into the threads that dequantise it, four rows a thread in flight
//      (the copy engine spends ~7 ns a row, which a tile's 128 separate rows
//      turn into the longest step), the next tile's rows prefetched into L2;
//      the rows are dequantised into shared memory as fp16 R[t][c] in
//      128-byte-swizzled blocks of 64 channels. fp16 holds every row value
//      exactly: an E2M1 x E4M3 product has at most 6 significant bits and
//      lies in [2^-10, 2688]; an E4M3 SWA value is a subset of fp16;
//   2. S^T[t][h] = R[t] . Q[h] on the tensor cores (kind::f16, M = 128 rows,
//      N = 64 heads, K = 512). Q was converted once per CTA from bf16 to fp16
//      with a power-of-two scale per head (2^k_h puts the head's largest
//      |q| in [2^14, 2^15)); this is exact for every value above 2^-17 of
//      that maximum, and S is multiplied back by 2^-k_h in the softmax;
//   3. per-head max and sum over the tile's rows (four lane-quadrant warps
//      per group of 16 heads meet at a named barrier); P = 2^(S log2 e - m)
//      rounded to fp16 (relative error <= 2^-11, against the 2^-9 of bf16)
//      and stored as the K-major B operand;
//   4. O^T[c][h] = sum_t R[t][c] P[h][t] on the tensor cores (M = 128
//      channels x 4 blocks, N = 64, K = 128), the R tile read as an MN-major
//      operand; the unnormalised O is staged in shared memory and sent to the
//      workspace by one bulk copy, (m, l) by plain stores.
// The SWA tiles depend on nothing the kernel before this one writes, so they
// run before the programmatic-launch wait; only the selected tiles follow it.
// Merge: after one cluster barrier (release / acquire) CTA r bulk-copies the
// slices of heads [64r/C, 64(r+1)/C) of every partial from the workspace
// (L2), weighs them by 2^(m_j - M) / L in fixed partial order
// (deterministic) and writes the output and the log-sum-exp.
#pragma once

#include "tc_common.cuh"

namespace csa2 {
namespace attn_tc {

constexpr int kThreads = 512;                   // 16 warps: 4 TMEM lane quadrants x 4
constexpr int kRows = 128;                      // rows per tile (M)
constexpr int kMaxCluster = 8;                  // CTAs of one query (portable cluster size)
constexpr int kBlkR = kRows * 128;              // one 64-channel block of R: [128 t][128 B] = 16 KiB
constexpr int kQBlk = kHeads * 128;             // one 64-channel block of Q: [64 h][128 B] = 8 KiB
constexpr int kPBlk = kHeads * 128;             // 64 rows of P: [64 h][128 B] = 8 KiB
constexpr int kOffR = 0;                        // 8 blocks = 128 KiB
constexpr int kOffQ = kOffR + 8 * kBlkR;        // 8 blocks = 64 KiB
constexpr int kOffP = kOffQ + 8 * kQBlk;        // 2 blocks = 16 KiB
constexpr int kOffMisc = kOffP + 2 * kPBlk;
constexpr int kOffStage = kOffR + 4 * kBlkR;    // an SWA tile's raw rows, in R's upper half (64 KiB)
constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;                   // S^T: 64 columns (heads), lanes = rows
constexpr uint32_t kColO = 64;                  // O^T: 4 blocks x 64 columns (heads), lanes = channels
constexpr int kMaxPartials = 36;                // 32 tiles of selected rows (k <= 4096) + 4 SWA tiles (<= 512 rows)

// the kernel's static arrays take under 10 KiB (8.5 KiB at most over the modes)
static_assert(kSmemBytes <= 232448 - 10240, "shared memory budget (static arrays included)");
static_assert(kRows * kHeadDim <= 4 * kBlkR, "the SWA staging fits in R's upper half");
// merge: (max, sum) and weights of every partial of the CTA's heads live in
// the P region (at most 36 partials x 16 heads with 4 or more CTAs, 5 x 64
// with one CTA, 6 x 32 with two, 7 x 22 with three)
static_assert(36 * 16 * 12 <= 2 * kPBlk && 7 * 22 * 12 <= 2 * kPBlk, "merge scratch fits the P region");

// kind::f16 with fp16 A/B, fp32 accumulate; a_mn / b_mn select MN-major operands.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t M, uint32_t N, uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4)  // D format: f32 (A and B format fields 0: f16)
         | (a_mn & 1u) << 15 | (b_mn & 1u) << 16 | ((N >> 3) & 63u) << 17 | ((M >> 4) & 31u) << 24;
}

__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Two E4M3 bytes (bits 0..7 and 8..15) to two fp16 values (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(r) : "r"(two));
  return r;
}

// Two fp32 values to one fp16x2 word (`lo` in bits 0..15), round to nearest even.
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight E2M1 codes (the 32-bit w: channel i in bits 4i..4i+3) to eight exact
// fp16 values in four fp16x2 words (o0: channels 0, 1; ...; o3: 6, 7).
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t w, uint32_t& o0, uint32_t& o1, uint32_t& o2, uint32_t& o3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(w));
}

// Transpose-reduce across a warp: lane L holds v[0..16) (one value per head);
// afterwards lane L returns the reduction over all 32 lanes of head L mod 16.
// v is overwritten.
template <bool kMax>
__device__ __forceinline__ float warp_transpose_reduce16(float (&v)[16], int lane) {
#pragma unroll
  for (int width = 8; width >= 1; width >>= 1) {
    const bool up = (lane & width) != 0;
#pragma unroll
    for (int i = 0; i < width; ++i) {
      const float keep = up ? v[i + width] : v[i];
      const float send = up ? v[i] : v[i + width];
      const float got = __shfl_xor_sync(0xffffffffu, send, width);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  const float o = __shfl_xor_sync(0xffffffffu, v[0], 16);
  return kMax ? fmaxf(v[0], o) : v[0] + o;
}

// 2^x (ex2.approx: relative error below 2^-22; +inf/-inf/NaN pass through).
__device__ __forceinline__ float fast_exp2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Sequential mode: the reference max a head's P is taken against (log2
// domain). It stays at the running value `ref` until a tile's max `mt` passes
// it by more than kSeqMaxSlack, so that most tiles leave O^T as it is: P is
// then at most 2^kSeqMaxSlack, far inside fp16, and the output O / l and the
// log-sum-exp are the same quantities whatever reference is used.
constexpr float kSeqMaxSlack = 8.0f;
__device__ __forceinline__ float seq_ref_max(float ref, float mt) {
  return mt > ref + kSeqMaxSlack ? mt : ref;
}

// A hint: the cache line holding p is fetched into L2.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// (max, sum) pair into the shared memory of CTA `rank` of the cluster.
__device__ __forceinline__ void st_cluster_f32x2(const void* local_addr, uint32_t rank, float x, float y) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(tc::smem_u32(local_addr)), "r"(rank));
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(remote), "f"(x), "f"(y) : "memory");
}

__device__ __forceinline__ void cluster_sync_release_acquire() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Modes: the tiles of a query spread over a cluster and merged through the
// workspace (latency: every tile in parallel), one sequence's Reuse layers in
// a cluster, or a query's tiles in sequence on one CTA (throughput).
enum : int { kModeCluster = 0, kModeReuse = 1, kModeSeq = 2 };

// grid (C, units of the launch), clusters of C CTAs along x. A unit is one
// query (kModeCluster, kModeSeq) or one sequence with its L Reuse layers
// (kModeReuse).
//
// Reuse mode ("DeepSeek-V4.1-Flash" section 2.3.1: the Reuse layers attend
// to the Full layer's selection with their own Q and SWA rows): a cluster
// serves a sequence. Its work items are the L x n_swt SWA tiles (one layer
// each) and the n_sel tiles of selected rows, each gathered and dequantised
// once and then attended by the L layers back to back while the next layer's
// Q is being loaded. Partials are written to the workspace by plain stores,
// and the cluster merges the L x 64 (layer, head) rows.
//
// Sequential mode (C = 1, for launches that fill the device several times
// over): the CTA walks its query's tiles in turn with an online softmax: the
// running (max, sum) of each head lives in shared memory, O^T stays in tensor
// memory and is rescaled by 2^(m_old - m_new) before each tile's PV product
// accumulates onto it, and the CTA writes the normalised output itself, with
// no partials and no merge.
template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, AttnArgs a) {
  constexpr bool kReuse = kMode == kModeReuse;
  constexpr bool kSeq = kMode == kModeSeq;
  // barriers, tensor memory, Q and the SWA tiles need nothing from the
  // preceding kernel; its outputs (the indices) are read after pdl_wait()
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = tc::smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  uint8_t* sR = sm + kOffR;
  uint8_t* sQ = sm + kOffQ;
  uint8_t* sP = sm + kOffP;
  uint8_t* sStage = sm + kOffStage;
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(sm + kOffMisc);  // S^T complete
  uint64_t* bar_pv = bar_s + 1;                                  // O^T complete
  uint64_t* q_full = bar_s + 2;                                  // Q landed
  uint64_t* bar_g = bar_s + 3;                                   // a tile's rows landed (128 arrivals)
  uint64_t* bar_m = bar_s + 4;                                   // merge slices landed
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + kOffMisc + 40);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + kOffMisc + 44);
  __shared__ __align__(16) float red_m[4][kHeads];
  __shared__ __align__(16) float red_l[4][kHeads];
  __shared__ float q_mul[kHeads];        // sm_scale * 2^-k_h * log2(e)
  __shared__ int row_valid[kRows];       // 0 none, 1 selected latent, 2 SWA row
  __shared__ int64_t row_src[kRows];     // a selected tile's cache row per tile row (-1: none)
  // (max, sum) of every partial for the (layer,) head rows this CTA merges,
  // written by the CTAs of the cluster through distributed shared memory:
  // [part][row - hb0]
  __shared__ float2 ml_in[kMaxPartials * 16];
  // sequential mode: running max (log2 domain) and sum of each head, and the
  // factor this tile rescales O by
  __shared__ float m_run[kHeads], l_run[kHeads], alpha_s[kHeads];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = (int)gridDim.x;
  const int rank = (int)blockIdx.x;
  const int unit = a.q0 + (int)blockIdx.y;   // query, or sequence in Reuse mode
  const int L = kReuse ? a.L : 1;
  const int seq = kReuse ? unit : unit / a.L;
  const int HR = kHeads * L;                 // (layer, head) rows of the unit
  const int n_swt = a.n_swt, n_sel = a.n_sel, n_part = a.n_part;
  // Reuse mode: a selected tile is one item per group of lgrp layers (gathered
  // once per group); SWA tiles are one item per layer
  const int lgrp = kReuse ? a.lgrp : 1;
  const int n_grp = L / lgrp;
  const int n_items = L * n_swt + n_sel * n_grp;   // SWA tiles (per layer), then (selected tile, group)
  // partial rows of the unit in the workspace: [layer][n_part][16][64][32]
  float* part_o_u = a.part_o + (int64_t)blockIdx.y * L * n_part * kHeads * kHeadDim;

  if (kSeq && tid < kHeads) {
    m_run[tid] = -INFINITY;
    l_run[tid] = 0.0f;
  }
  if (tid == 0) {
    tc::mbar_init(bar_s, 1);
    tc::mbar_init(bar_pv, 1);
    tc::mbar_init(q_full, 1);
    tc::mbar_init(bar_g, kRows);
    tc::mbar_init(bar_m, 1);
    *s_abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(s_tmem, kTmemCols);
  // every CTA of the cluster has started before any writes into another's
  // shared memory (the wait follows the first Q conversion)
  cluster_arrive_relaxed();
  __syncthreads();

  // the layer of each attention pass of this CTA, in order: an SWA item is one
  // pass of its layer, a selected item one pass per layer
  auto item_layer0 = [&](const int j) {
    if (!kReuse) return 0;
    return j < L * n_swt ? j / n_swt : ((j - L * n_swt) % n_grp) * lgrp;
  };
  // Q of query (seq, layer) into sQ: 8 TMA boxes of [64 h][64 c] bf16, 128-byte swizzle
  auto issue_q = [&](const int layer) {
    if (tid == 0) {
      const int qrow = (kReuse ? seq * L + layer : unit) * kHeads;
      tc::mbar_arrive_expect_tx(q_full, 8 * kQBlk);
      for (int b = 0; b < 8; ++b) tc::tma_load_2d(sQ + b * kQBlk, &tmap_q, b * 64, qrow, q_full);
    }
  };
  uint32_t q_loads = 0;   // parity source of q_full
  int q_layer = -1;       // layer whose Q sQ holds (or is loading)
  if (rank < n_items) {
    q_layer = item_layer0(rank);
    issue_q(q_layer);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;

  // ---- Q to fp16 with a power-of-two scale per head: thread (h, j) owns the
  // 16-byte column j of head h's row in each of the 8 blocks (bank-conflict
  // free: the 8 threads of a head cover the row's 8 columns) ----
  auto convert_q = [&]() {
    const bool ok = __all_sync(0xffffffffu, tc::mbar_wait_bounded(q_full, q_loads & 1u, s_abort, &g_attn_error));
    ++q_loads;
    const int h = tid >> 3, j = tid & 7;
    const uint32_t col = (uint32_t)((j ^ (h & 7)) << 4);
    uint4 v[8];
#pragma unroll
    for (int b = 0; b < 8; ++b)
      v[b] = ok ? *reinterpret_cast<const uint4*>(sQ + b * kQBlk + h * 128 + col) : make_uint4(0u, 0u, 0u, 0u);
    uint32_t amax = 0;   // bf16 bits of |q| compare as unsigned integers
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const uint32_t w[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) amax = max(amax, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
    }
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    // largest |q| has exponent e (bf16 exponent field e + 127); 2^(14 - e) puts
    // it in [2^14, 2^15). Clamped so that 2^k and 2^-k stay normal fp32.
    int k = 0;
    if (amax != 0u) {
      const int e = (int)((amax >> 7) & 0xFFu) - 127;
      k = min(max(14 - e, -100), 100);
    }
    const float up = __int_as_float((127 + k) << 23);
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const uint32_t w[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        o[i] = f32x2_to_f16x2(__uint_as_float(w[i] << 16) * up, __uint_as_float(w[i] & 0xFFFF0000u) * up);
      *reinterpret_cast<uint4*>(sQ + b * kQBlk + h * 128 + col) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (j == 0) q_mul[h] = a.sm_scale * __int_as_float((127 - k) << 23) * 1.4426950408889634f;
    // the converted Q is read by the MMA (async proxy) after the next barrier
    tc::fence_proxy_async_smem();
  };
  bool q_ready = false;   // sQ holds the converted Q of q_layer
  if (rank < n_items) {
    convert_q();
    q_ready = true;
  }

  cluster_wait();   // the peers have started: their shared memory may be written
  uint32_t items_done = 0;   // parity source of bar_g
  uint32_t passes_done = 0;  // parity source of bar_s / bar_pv

  // ---- one tile's rows: rows [128 tile, 128 tile + 128) of the SWA window of
  // query qi_swa (swa: one bulk copy) or of the sequence's selected list
  // (plain loads by the dequantising threads), dequantised into R ----
  // thread r < 128: the index of row r of the CTA's next selected tile, loaded
  // while the current tile is attended (pf_tile: that tile, -1 none); the
  // sequence's visible count, read once
  int32_t pf_idx = -1;
  int pf_tile = -1;
  int64_t nv_seq = -1;
  bool pf_rows = false;   // pf_idx's row is still to be prefetched into L2
  auto gather_dequant = [&](const bool swa, const int tile, const int qi_swa, const int next_sel_tile) {
    const uint32_t par = items_done & 1u;
    // SWA tiles: one contiguous bulk copy of the tile's rows into the staging
    // area. Selected tiles: thread r < 128 resolves row r to its cache row,
    // and the dequantising threads load the codes and scales straight from
    // global memory (no staging copy, no wait on the copy engine)
    if (tid < kRows) {
      int valid = 0;
      int64_t src = 0;
      const int t = tile * kRows + tid;
      if (swa) {
        // in prefill, row t of query qi is row qi + t of the array, and rows
        // before swa_first_row lie before a Bounded Replay start
        if (t < a.n_swa && (int64_t)qi_swa + t >= (int64_t)a.swa_first_row) valid = 2;
        if (tid == 0) {
          const int n_rows = min(kRows, a.n_swa - tile * kRows);
          const uint32_t bytes = (uint32_t)n_rows * kHeadDim;
          tc::mbar_arrive_expect_tx(bar_g, bytes);
          tc::bulk_load(sStage, a.swa + (int64_t)qi_swa * a.swa_q_stride + (int64_t)tile * kRows * kHeadDim, bytes,
                        bar_g);
        } else {
          tc::mbar_arrive(bar_g);
        }
      } else {
        if (t < a.k) {
          // n_visible may come from the kernel before this one (a KV append):
          // read after pdl_wait(), like the indices
          if (nv_seq < 0) nv_seq = a.n_visible ? (int64_t)a.n_visible[seq] : a.nv_const;
          const int32_t p = pf_tile == tile ? pf_idx : a.idx[(int64_t)seq * a.k + t];
          if (p >= 0) {
            if (p < nv_seq) {
              valid = 1;
              src = (int64_t)seq * a.kv_seq_stride + p;
            } else {
              record_error(&g_attn_error, CSA2_ERR_DEVICE);
            }
          }
        }
        row_src[tid] = valid ? src : -1;
        // the next selected tile's index for this row, in flight through this tile
        if (next_sel_tile >= 0) {
          const int tn = next_sel_tile * kRows + tid;
          pf_idx = tn < a.k ? a.idx[(int64_t)seq * a.k + tn] : -1;
          pf_tile = next_sel_tile;
        }
      }
      row_valid[tid] = valid;
    }
    __syncthreads();
    bool g_ok = true;
    if (swa) {
      g_ok = __all_sync(0xffffffffu, tc::mbar_wait_bounded(bar_g, par, s_abort, &g_attn_error));
      ++items_done;
    }
    // ---- dequantise into R (fp16, SW128 blocks of 64 channels). The staged
    // SWA bytes sit in R's upper half: read them all, then write R ----
    if (swa) {
      // warp w: rows 8w .. 8w+7; lane l: channels 16l .. 16l+15 of the row
      uint4 raw[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = warp * 8 + i;
        raw[i] = (g_ok && row_valid[r]) ? *reinterpret_cast<const uint4*>(sStage + r * kHeadDim + lane * 16)
                                        : make_uint4(0u, 0u, 0u, 0u);
      }
      __syncthreads();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = warp * 8 + i;
        uint8_t* blk = sR + (lane >> 2) * kBlkR;
        const uint32_t c0 = (uint32_t)(lane & 3) * 2u;
        // lanes of odd blocks write their second chunk first, so that the
        // lanes of one store cover eight different bank groups
        const uint32_t sw = (uint32_t)(lane >> 2) & 1u;
        const uint4 e = raw[i];
        const uint32_t a0 = sw ? e.z : e.x, a1 = sw ? e.w : e.y, b0 = sw ? e.x : e.z, b1 = sw ? e.y : e.w;
        // zero bytes decode to +0: invalid rows stay zero (P = 0 must not meet NaN)
        *reinterpret_cast<uint4*>(blk + tc::sw128_offset((uint32_t)r, c0 + sw)) =
            make_uint4(e4m3x2_to_f16x2(a0 & 0xFFFFu), e4m3x2_to_f16x2(a0 >> 16), e4m3x2_to_f16x2(a1 & 0xFFFFu),
                       e4m3x2_to_f16x2(a1 >> 16));
        *reinterpret_cast<uint4*>(blk + tc::sw128_offset((uint32_t)r, c0 + (sw ^ 1u))) =
            make_uint4(e4m3x2_to_f16x2(b0 & 0xFFFFu), e4m3x2_to_f16x2(b0 >> 16), e4m3x2_to_f16x2(b1 & 0xFFFFu),
                       e4m3x2_to_f16x2(b1 >> 16));
      }
    } else {
      // warp w: rows 8w .. 8w+7, two per step; lane l: row 8w + 2i + l / 16,
      // channels 32 (l % 16) .. +31 (16 bytes of codes, 2 scale bytes)
      uint4 raw[4];
      uint32_t scl[4];
      const int c16 = lane & 15;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t src = row_src[warp * 8 + 2 * i + (lane >> 4)];
        raw[i] = src >= 0 ? __ldg(reinterpret_cast<const uint4*>(a.kv_data + src * kKvBytes) + c16)
                          : make_uint4(0u, 0u, 0u, 0u);
        scl[i] = src >= 0 ? (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(a.kv_scale + src * kKvScales) + c16)
                          : 0u;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = warp * 8 + 2 * i + (lane >> 4);
        uint8_t* blk = sR + (c16 >> 1) * kBlkR;
        const uint32_t c0 = (uint32_t)(c16 & 1) * 4u;
        const uint32_t sc2 = e4m3x2_to_f16x2(scl[i]);       // scales of channels +0..15 (low) and +16..31 (high)
        const uint32_t sa = __byte_perm(sc2, 0u, 0x1010u);  // low scale in both halves
        const uint32_t sb = __byte_perm(sc2, 0u, 0x3232u);  // high scale in both halves
        // word k of the 16 bytes: channels 8k .. 8k+7; step kq writes word
        // (kq + c16 / 2) % 4, so that the 16 lanes of a row cover eight bank
        // groups
        const int rot = (c16 >> 1) & 3;
#pragma unroll
        for (int kq = 0; kq < 4; ++kq) {
          const int k = (kq + rot) & 3;
          const uint32_t w = k == 0 ? raw[i].x : k == 1 ? raw[i].y : k == 2 ? raw[i].z : raw[i].w;
          const uint32_t s2 = k < 2 ? sa : sb;
          uint32_t o0, o1, o2, o3;
          e2m1x8_to_f16(w, o0, o1, o2, o3);
          // zero codes with a zero scale give +0: invalid rows stay zero
          *reinterpret_cast<uint4*>(blk + tc::sw128_offset((uint32_t)r, c0 + (uint32_t)k)) =
              make_uint4(mul_f16x2(o0, s2), mul_f16x2(o1, s2), mul_f16x2(o2, s2), mul_f16x2(o3, s2));
        }
      }
      // the next selected tile's row for this thread (its index arrived during
      // this tile) is brought into L2 while this tile is attended
      if (tid < kRows && next_sel_tile >= 0 && pf_tile == next_sel_tile && pf_idx >= 0 && pf_idx < nv_seq) {
        const int64_t nsrc = (int64_t)seq * a.kv_seq_stride + pf_idx;
        prefetch_l2(a.kv_data + nsrc * kKvBytes);
        prefetch_l2(a.kv_data + nsrc * kKvBytes + 128);
        prefetch_l2(a.kv_scale + nsrc * kKvScales);
      }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    return g_ok;
  };

  // ---- one attention pass over the rows in R with the converted Q of layer
  // `layer` in sQ, giving partial `part` of that layer's query. next_layer >= 0:
  // the layer of the CTA's next pass, whose Q is loaded into sQ as soon as
  // this pass's S^T is complete. more_rows: R is rewritten after this pass ----
  auto attend = [&](const int layer, const int part, const int next_layer, const bool more_rows) {
    const uint32_t par = passes_done & 1u;
    // ---- S^T = R Q^T ----
    if (tid == 0 && !*s_abort) {
      constexpr uint32_t idesc = idesc_f16(128, 64, 0, 0);
      // descriptors advance by constant steps (address fields count 16 bytes)
      const uint64_t ad0 = tc::smem_desc(tc::smem_u32(sR), 0, 1024, tc::kSwizzle128B);
      const uint64_t bd0 = tc::smem_desc(tc::smem_u32(sQ), 0, 1024, tc::kSwizzle128B);
#pragma unroll
      for (int i = 0; i < 32; ++i) {   // block b = i / 4 (64 channels), K step kk = i % 4 (16 channels)
        const uint64_t ko = (uint64_t)((i & 3) * 2);
        tc::mma_bf16(tmem + kColS, ad0 + (uint64_t)((i >> 2) * (kBlkR >> 4)) + ko,
                     bd0 + (uint64_t)((i >> 2) * (kQBlk >> 4)) + ko, idesc, i ? 1u : 0u);
      }
      tc::mma_commit(bar_s);
    }
    __syncwarp();
    const bool s_ok = __all_sync(0xffffffffu, !*s_abort && tc::mbar_wait_bounded(bar_s, par, s_abort, &g_attn_error));
    tc::tc_fence_after();
    // sQ is free once S^T is complete: start the next layer's Q
    if (kReuse && next_layer >= 0 && next_layer != q_layer) {
      issue_q(next_layer);
      q_layer = next_layer;
      q_ready = false;
    }
    // ---- softmax: warp w reads the 32 rows of lane quadrant w % 4 and the 16
    // heads 16 (w / 4) ..; the four quadrant warps of a head group meet at
    // named barrier 1 + w / 4 ----
    const int rq = warp & 3, hg = warp >> 2, h0 = hg * 16;
    const int row = rq * 32 + lane;
    const bool rv = s_ok && row_valid[row] != 0;
    float p[16];
    {
      uint32_t sr[16];
      if (s_ok) {
        tc::tmem_ld_32x32b_x16(tmem + ((uint32_t)(rq * 32) << 16) + kColS + (uint32_t)h0, sr);
        tc::tmem_ld_wait();
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) p[j] = rv ? __uint_as_float(sr[j]) * q_mul[h0 + j] : -INFINITY;
    }
    {
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = p[j];
      const float m = warp_transpose_reduce16<true>(v, lane);
      if (lane < 16) red_m[rq][h0 + lane] = m;
    }
    named_barrier(1 + hg, 128);
    float M[16];
#pragma unroll
    for (int j4 = 0; j4 < 4; ++j4) {
      float4 m4 = *reinterpret_cast<const float4*>(&red_m[0][h0 + 4 * j4]);
#pragma unroll
      for (int q = 1; q < 4; ++q) {
        const float4 o = *reinterpret_cast<const float4*>(&red_m[q][h0 + 4 * j4]);
        m4.x = fmaxf(m4.x, o.x);
        m4.y = fmaxf(m4.y, o.y);
        m4.z = fmaxf(m4.z, o.z);
        m4.w = fmaxf(m4.w, o.w);
      }
      M[4 * j4] = m4.x;
      M[4 * j4 + 1] = m4.y;
      M[4 * j4 + 2] = m4.z;
      M[4 * j4 + 3] = m4.w;
    }
    if (kSeq) {   // P relative to the head's reference max (seq_ref_max)
#pragma unroll
      for (int j = 0; j < 16; ++j) M[j] = seq_ref_max(m_run[h0 + j], M[j]);
    }
    // P = 2^(s - M), fp16, stored K-major for the PV product: row h of the
    // 64-row block row / 64, element row % 64
    {
      uint8_t* blkp = sP + (row >> 6) * kPBlk;
      const uint32_t chunk = (uint32_t)(row & 63) >> 3, within = ((uint32_t)row & 7u) * 2u;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        p[j] = (p[j] == -INFINITY) ? 0.0f : fast_exp2(p[j] - M[j]);
        const __half hv = __float2half_rn(p[j]);
        *reinterpret_cast<__half*>(blkp + tc::sw128_offset((uint32_t)(h0 + j), chunk) + within) = hv;
      }
    }
    {
      const float l = warp_transpose_reduce16<false>(p, lane);
      if (lane < 16) red_l[rq][h0 + lane] = l;
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (kSeq) {
      // running (max, sum) of each head; O^T of the earlier tiles rescaled to
      // the new max before this tile's PV accumulates onto it
      bool moved = false;
      if (tid < kHeads) {
        const int h = tid;
        const float mt = fmaxf(fmaxf(red_m[0][h], red_m[1][h]), fmaxf(red_m[2][h], red_m[3][h]));
        const float mo = m_run[h], mn = seq_ref_max(mo, mt);
        moved = mn != mo;
        const float alpha = !moved ? 1.0f : mo == -INFINITY ? 0.0f : fast_exp2(mo - mn);
        const float lt = s_ok ? red_l[0][h] + red_l[1][h] + red_l[2][h] + red_l[3][h] : 0.0f;
        l_run[h] = l_run[h] * alpha + lt;
        m_run[h] = mn;
        alpha_s[h] = alpha;
      }
      // O^T of the earlier tiles is rescaled only when some head's reference
      // max moved (the barrier also publishes alpha_s)
      if (__syncthreads_or(moved) && passes_done > 0) {
        const uint32_t o_base = tmem + ((uint32_t)(rq * 32) << 16) + kColO + 64u * (uint32_t)(warp >> 2);
#pragma unroll 1
        for (int hh = 0; hh < kHeads; hh += 16) {
          uint32_t ov[16];
          tc::tmem_ld_32x32b_x16(o_base + (uint32_t)hh, ov);
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha_s[hh + j]);
          tc::tmem_st_32x32b_x16(o_base + (uint32_t)hh, ov);
        }
        tc::tmem_st_wait();
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();
      }
    }
    if (pf_rows) {   // (only threads below 128 set it)
      if (pf_idx >= 0 && pf_idx < nv_seq) {
        const int64_t nsrc = (int64_t)seq * a.kv_seq_stride + pf_idx;
        prefetch_l2(a.kv_data + nsrc * kKvBytes);
        prefetch_l2(a.kv_data + nsrc * kKvBytes + 128);
        prefetch_l2(a.kv_scale + nsrc * kKvScales);
      }
      pf_rows = false;
    }
    // ---- O^T = R^T P^T : 4 x (M = 128 channels), N = 64, K = 128 rows ----
    if (tid == 0 && s_ok) {
      constexpr uint32_t idesc = idesc_f16(128, 64, 1, 0);  // A (channels x rows) is MN-major
      // A: channels 128 mb .. +127 (64-channel blocks 2mb, 2mb+1: LBO apart),
      //    rows 16 kk .. +15 (8-row groups: SBO apart);
      // B: the 64 P rows (heads), rows t = 16 kk .. +15 inside the 64-row block kk / 4
      const uint64_t ad0 = tc::smem_desc(tc::smem_u32(sR), kBlkR, 1024, tc::kSwizzle128B);
      const uint64_t bd0 = tc::smem_desc(tc::smem_u32(sP), 0, 1024, tc::kSwizzle128B);
#pragma unroll
      for (int i = 0; i < 4 * (kRows / 16); ++i) {   // channel block mb = i / 8, K step kk = i % 8
        const int mb = i >> 3, kk = i & 7;
        tc::mma_bf16(tmem + kColO + 64u * (uint32_t)mb,
                     ad0 + (uint64_t)((2 * mb * kBlkR + kk * 16 * 128) >> 4),
                     bd0 + (uint64_t)(((kk >> 2) * kPBlk + (kk & 3) * 32) >> 4), idesc,
                     (kk || (kSeq && passes_done > 0)) ? 1u : 0u);
      }
      tc::mma_commit(bar_pv);
    }
    // (m, l) of the pass, log2 domain (l = 0 marks a partial with no rows),
    // into the shared memory of the CTA that merges (layer, head) row hr
    if (!kSeq && tid < kHeads) {
      const int h = tid, hr = layer * kHeads + h;
      const float m = fmaxf(fmaxf(red_m[0][h], red_m[1][h]), fmaxf(red_m[2][h], red_m[3][h]));
      const float l = s_ok ? red_l[0][h] + red_l[1][h] + red_l[2][h] + red_l[3][h] : 0.0f;
      int r = (hr * C) / HR;   // owner: the rank r with HR r / C <= hr < HR (r + 1) / C
      while (HR * (r + 1) / C <= hr) ++r;
      while (HR * r / C > hr) --r;
      const int o0 = HR * r / C, onh = HR * (r + 1) / C - o0;
      st_cluster_f32x2(&ml_in[part * onh + (hr - o0)], (uint32_t)r, m, l);
    }
    __syncwarp();
    const bool ok = __all_sync(0xffffffffu, s_ok && tc::mbar_wait_bounded(bar_pv, par, s_abort, &g_attn_error));
    tc::tc_fence_after();
    // ---- partial O: warp w reads the 32 channel lanes 32 cb .. of quadrant
    // w % 4 in block w / 4 (cb = 4 (w / 4) + w % 4), all 64 heads; a partial is
    // laid out [cb][h][32] ----
    if (!kSeq) {
      const int cb = (warp >> 2) * 4 + rq;
      const uint32_t o_base = tmem + ((uint32_t)(rq * 32) << 16) + kColO + 64u * (uint32_t)(warp >> 2);
      float* dst = part_o_u + (((int64_t)layer * n_part + part) * 16 + cb) * (kHeads * 32);
      if (kReuse) {
        // R stays for the next layer: plain stores, 128 contiguous bytes per
        // warp and head
#pragma unroll
        for (int hh = 0; hh < kHeads; hh += 32) {
          uint32_t ov[32];
          if (ok) {
            tc::tmem_ld_32x32b_x32(o_base + (uint32_t)hh, ov);
            tc::tmem_ld_wait();
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) dst[(hh + j) * 32 + lane] = ok ? __uint_as_float(ov[j]) : 0.0f;
        }
      } else {
        // staged in R as [h][32] fp32, then 8 KiB to the workspace by one bulk copy
        float* so = reinterpret_cast<float*>(sR) + cb * (kHeads * 32);
#pragma unroll
        for (int hh = 0; hh < kHeads; hh += 32) {
          uint32_t ov[32];
          if (ok) {
            tc::tmem_ld_32x32b_x32(o_base + (uint32_t)hh, ov);
            tc::tmem_ld_wait();
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) so[(hh + j) * 32 + lane] = ok ? __uint_as_float(ov[j]) : 0.0f;
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tc::bulk_store(dst, so, kHeads * 32 * 4);
          tc::bulk_commit();
          if (more_rows) tc::bulk_wait_read_all();   // R is rewritten by the next tile
        }
      }
    }
    tc::tc_fence_before();
    ++passes_done;
    // the next pass rewrites S, P, O (and maybe R) only after every thread is
    // past this pass's reads of them
    __syncthreads();
  };

  // items j of the list [SWA tiles, selected tiles] belong to CTA j mod C; the
  // SWA tiles come first, before the wait for the indices
  bool waited = false;
#pragma unroll 1
  for (int j = rank; j < n_items; j += C) {
    const bool swa = j < L * n_swt;
    if (!swa && !waited) {
      pdl_wait();
      waited = true;
    }
    const int jn = j + C;   // the CTA's next item
    const int l0 = item_layer0(j);
    const int swa_tile = swa ? j - l0 * n_swt : 0;
    const int sel_tile = swa ? 0 : (j - L * n_swt) / n_grp;
    const int next_sel = jn < n_items && jn >= L * n_swt ? (jn - L * n_swt) / n_grp : -1;
    const bool rows_ok =
        gather_dequant(swa, swa ? swa_tile : sel_tile, kReuse ? seq * L + l0 : unit, swa ? -1 : next_sel);
    (void)rows_ok;
    if (!kSeq && swa && next_sel >= 0 && !waited) {
      // the CTA's next item is a selected tile: wait for the indices now, so
      // that this thread's index of it arrives (and its row is prefetched into
      // L2, pf_rows) while the SWA tile is attended. (Not in the sequential
      // mode: there the SWA pass of a launch's first CTAs overlaps the end of
      // the launch before, which an earlier wait would give up.)
      pdl_wait();
      waited = true;
      if (tid < kRows) {
        if (nv_seq < 0) nv_seq = a.n_visible ? (int64_t)a.n_visible[seq] : a.nv_const;
        const int tn = next_sel * kRows + tid;
        pf_idx = tn < a.k ? a.idx[(int64_t)seq * a.k + tn] : -1;
        pf_tile = next_sel;
        pf_rows = true;
      }
    }
    const int n_layers = swa ? 1 : lgrp;
    for (int li = 0; li < n_layers; ++li) {
      const int layer = l0 + li;
      if (!q_ready || q_layer != layer) {   // its load was started by the previous pass (or now)
        if (q_layer != layer) {
          issue_q(layer);
          q_layer = layer;
        }
        convert_q();
        q_ready = true;
        __syncthreads();
      }
      const int next_layer = li + 1 < n_layers ? layer + 1 : (jn < n_items ? item_layer0(jn) : -1);
      attend(layer, swa ? swa_tile : n_swt + sel_tile, next_layer, jn < n_items);
    }
  }
  if (!waited) pdl_wait();

  if (kSeq) {
    // ---- output: O^T / l per head from tensor memory; warp w: channels
    // 128 (w / 4) + 32 (w % 4) + lane, all 64 heads ----
    const int rq = warp & 3;
    const int c = 128 * (warp >> 2) + 32 * rq + lane;
    if (tid < kHeads) {
      const float l = l_run[tid];
      alpha_s[tid] = l > 0.0f ? 1.0f / l : 0.0f;
      if (a.lse) a.lse[(int64_t)unit * kHeads + tid] = l > 0.0f ? (m_run[tid] + log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t o_base = tmem + ((uint32_t)(rq * 32) << 16) + kColO + 64u * (uint32_t)(warp >> 2);
    float* of = a.out_f32 ? a.out_f32 + (int64_t)unit * kHeads * kHeadDim + c : nullptr;
    uint16_t* ob = a.out + (int64_t)unit * kHeads * kHeadDim + c;
#pragma unroll 1
    for (int hh = 0; hh < kHeads; hh += 16) {
      uint32_t ov[16];
      if (passes_done > 0) {
        tc::tmem_ld_32x32b_x16(o_base + (uint32_t)hh, ov);
        tc::tmem_ld_wait();
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float v = passes_done > 0 ? __uint_as_float(ov[j]) * alpha_s[hh + j] : 0.0f;
        if (of) of[(hh + j) * kHeadDim] = v;
        ob[(hh + j) * kHeadDim] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
      }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      tc::tc_fence_after();
      tc::tmem_dealloc(tmem, kTmemCols);
    }
    return;
  }

  // ---- merge: rank r sums rows [HR r/C, HR (r+1)/C) over all partials ----
  if (kReuse) {
    // this CTA's partial stores are visible to the cluster after the barrier;
    // the merge reads them with bulk copies (async proxy)
    tc::fence_proxy_async_all();
  } else if (lane == 0) {
    tc::bulk_wait_all();       // this warp's partial slices are in global memory
    tc::fence_proxy_async_all();
  }
  __syncwarp();
  cluster_sync_release_acquire();
  if (kReuse) tc::fence_proxy_async_all();
  const int hb0 = HR * rank / C, hb1 = HR * (rank + 1) / C;
  const int nh = hb1 - hb0;
  // groups of up to 16 rows of one layer: the group's slices of the partials
  // come by bulk copies into R and Q (free now), a slot per partial laid out
  // [cb][gh][32]; each thread sums 4 float4 items in fixed partial order. The
  // first batch is requested before the weights are formed.
  auto group_size = [&](const int g0) { return min(min(16, nh - g0), kHeads - (hb0 + g0) % kHeads); };
  auto issue_batch = [&](const int g0, const int gh, const int j0, const int nb) {
    const uint32_t piece = (uint32_t)gh * 32 * 4;
    const int layer = (hb0 + g0) / kHeads, h0 = (hb0 + g0) % kHeads;
    if (tid == 0) tc::mbar_arrive_expect_tx(bar_m, (uint32_t)nb * 16 * piece);
    __syncwarp();
    if (tid < 16 * nb) {   // thread t copies piece cb = t % 16 of partial j0 + t / 16
      const int u = tid >> 4, cb = tid & 15;
      tc::bulk_load(sR + (size_t)u * 16 * piece + (size_t)cb * piece,
                    part_o_u + ((((int64_t)layer * n_part + j0 + u) * 16 + cb) * kHeads + h0) * 32, piece, bar_m);
    }
  };
  auto batch_size = [&](const int gh) { return (int)((uint32_t)(kOffP - kOffR) / ((uint32_t)gh * 32 * 4 * 16)); };
  if (nh > 0 && n_part > 0) issue_batch(0, group_size(0), 0, min(batch_size(group_size(0)), n_part));
  float* wts = reinterpret_cast<float*>(sP);   // [n_part][nh] weights
  __shared__ float lse_s[kHeads];
  // lse_s, wts: this CTA's rows (nh <= 64 when the plan allows this launch)
  if (tid < nh) {
    float M = -INFINITY;
    for (int j = 0; j < n_part; ++j)
      if (ml_in[j * nh + tid].y > 0.0f) M = fmaxf(M, ml_in[j * nh + tid].x);
    float Lsum = 0.0f;
    for (int j = 0; j < n_part; ++j) {   // fixed order
      const float2 ml = ml_in[j * nh + tid];
      const float e = ml.y > 0.0f ? fast_exp2(ml.x - M) : 0.0f;
      wts[j * nh + tid] = e;
      Lsum += ml.y * e;
    }
    const float inv = Lsum > 0.0f ? 1.0f / Lsum : 0.0f;
    for (int j = 0; j < n_part; ++j) wts[j * nh + tid] *= inv;
    lse_s[tid] = Lsum > 0.0f ? (M + log2f(Lsum)) * 0.6931471805599453f : -INFINITY;
  }
  // output row of (layer, head) row hr
  auto out_row = [&](const int hr) {
    return ((int64_t)(kReuse ? seq * L + hr / kHeads : unit) * kHeads + hr % kHeads);
  };
  if (a.lse && tid < nh) a.lse[out_row(hb0 + tid)] = lse_s[tid];
  uint32_t mpar = 0;
#pragma unroll 1
  for (int g0 = 0; g0 < nh;) {
    const int gh = group_size(g0);
    const uint32_t slot_bytes = (uint32_t)gh * 32 * 4 * 16;
    const int per_batch = batch_size(gh);
    float4 acc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int j0 = 0; j0 < n_part; j0 += per_batch) {
      const int nb = min(per_batch, n_part - j0);
      __syncthreads();   // the slots are free; the weights are visible
      if (g0 > 0 || j0 > 0) issue_batch(g0, gh, j0, nb);
      const bool m_ok = tc::mbar_wait_bounded(bar_m, mpar, s_abort, &g_attn_error);
      mpar ^= 1u;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int it = tid + u * kThreads;   // item: row g0 + it / 128, channels 4 (it % 128) ..
        if (it >= gh * (kHeadDim / 4)) break;
        const int hl = it >> 7, cb = (it >> 3) & 15, c4 = it & 7;
        const int off = ((cb * gh + hl) * 32 + 4 * c4) * 4;
#pragma unroll 1
        for (int jj = 0; jj < nb; ++jj) {   // fixed partial order
          const float4 v = m_ok ? *reinterpret_cast<const float4*>(sR + (size_t)jj * slot_bytes + off)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
          const float f = wts[(j0 + jj) * nh + g0 + hl];
          acc[u].x = fmaf(v.x, f, acc[u].x);
          acc[u].y = fmaf(v.y, f, acc[u].y);
          acc[u].z = fmaf(v.z, f, acc[u].z);
          acc[u].w = fmaf(v.w, f, acc[u].w);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int it = tid + u * kThreads;
      if (it >= gh * (kHeadDim / 4)) break;
      const int hl = it >> 7, c = (it & 127) * 4;
      const int64_t o = out_row(hb0 + g0 + hl) * kHeadDim + c;
      if (a.out_f32) *reinterpret_cast<float4*>(a.out_f32 + o) = acc[u];
      const __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[u].x, acc[u].y);
      const __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[u].z, acc[u].w);
      *reinterpret_cast<uint2*>(a.out + o) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1));
    }
    g0 += gh;
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
