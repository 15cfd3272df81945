// attention.cu -- sparse attention over the selected FP4 latents plus the FP8
// sliding window, for decode (B sequences x L layers sharing one Top-K) and
// prefill (T queries, each with its own Top-K and causal window).
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", section
// 2.3 (each Q attends to the selected entries together with the layer-local
// SWA KV), section 2.3.1 (Reuse layers reuse main KV and Top-K with their own
// Q and SWA KV), section 2.4.4 (FP4 main KV dequantised before attention; FP8
// SWA KV); mer.dev notes section 1 (64 heads of dim 512; the 512-dim KV latent
// is shared as K and V).
//
// Work split (attention_tc.cuh): the rows of a query are cut into tiles of
// 128 (SWA tiles, then selected tiles); a cluster of C CTAs serves one query,
// each tile gives a partial softmax, and the CTAs of the cluster merge the
// partials in fixed order, so results are deterministic.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace csa2 {

__device__ int g_attn_error = 0;

struct AttnArgs {
  const uint8_t* kv_data;   // plane base
  const uint8_t* kv_scale;
  int64_t kv_seq_stride;    // entries between sequences (0: one shared plane)
  const int32_t* n_visible; // per sequence, or null (then nv_const)
  int64_t nv_const;
  const int32_t* idx;       // [n_seq][k]
  int32_t k;
  int32_t L;                // queries per sequence (layers sharing the Top-K)
  int32_t lgrp;             // Reuse mode: layers attended per gather of a selected tile (divides L)
  const uint8_t* swa;       // SWA bytes
  int64_t swa_q_stride;     // bytes between consecutive queries' windows
  int32_t n_swa;
  int32_t swa_first_row;    // prefill: SWA rows before this row of the array are masked (Bounded Replay)
  float sm_scale;
  int32_t q0;               // first unit of this launch: query, or sequence in Reuse mode
  int32_t n_sel, n_swt, n_part;  // tiles of selected rows, SWA tiles, partials per query
  float* part_o;            // [units][L or 1][n_part][16][64][32]: unnormalised partial outputs, 32-channel blocks
  uint16_t* out;            // [n_q][64][512] bf16
  float* out_f32;           // nullable
  float* lse;               // nullable
};

}  // namespace csa2

#include "attention_tc.cuh"

using namespace csa2;

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

static constexpr int kQueriesPerLaunch = 256;  // bounds the workspace of one launch

int csa2_read_and_clear_attn_error(cudaStream_t s) {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_attn_error, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return CSA2_ERR_CUDA;
  if (cudaMemcpyToSymbolAsync(g_attn_error, &z, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return CSA2_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return CSA2_ERR_CUDA;
  return v;
}

// Opts the kernels into their dynamic shared memory, once per device.
static int attn_kernel_attr() {
  static Csa2PerDeviceOnce optin, optin_reuse, optin_seq;
  if (csa2_smem_optin((const void*)attn_tc::attn_tc_kernel<attn_tc::kModeCluster>, attn_tc::kSmemBytes, optin) !=
          CSA2_OK ||
      csa2_smem_optin((const void*)attn_tc::attn_tc_kernel<attn_tc::kModeSeq>, attn_tc::kSmemBytes, optin_seq) !=
          CSA2_OK)
    return CSA2_ERR_CUDA;
  return csa2_smem_optin((const void*)attn_tc::attn_tc_kernel<attn_tc::kModeReuse>, attn_tc::kSmemBytes, optin_reuse);
}

// How many clusters of `size` CTAs of the kernel (Reuse mode or not) can be
// resident at once (0: none), cached per device.
static int attn_max_clusters(int size, bool reuse = false) {
  constexpr int kMaxDevices = 64;
  static int cache[kMaxDevices][2][attn_tc::kMaxCluster + 1];  // count + 1; 0 unknown
  static std::mutex mu;
  int dev = 0;
  if (size < 1 || size > attn_tc::kMaxCluster) return 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(mu);
  int& slot = cache[dev][reuse ? 1 : 0][size];
  if (!slot) {
    int n = 0;
    if (attn_kernel_attr() == CSA2_OK) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)size, 1, 1);
      cfg.blockDim = dim3(attn_tc::kThreads);
      cfg.dynamicSmemBytes = attn_tc::kSmemBytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)size;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      const void* kern = reuse ? (const void*)attn_tc::attn_tc_kernel<attn_tc::kModeReuse>
                               : (const void*)attn_tc::attn_tc_kernel<attn_tc::kModeCluster>;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
      }
    }
    slot = n + 1;
  }
  return slot - 1;
}

struct AttnPlan {
  int n_sel, n_swt, n_part;  // tiles of selected rows, SWA tiles, partials per query
  int cluster;               // CTAs per query
  bool seq;                  // one CTA per query walking its tiles (online softmax, no partials)
};

// Tiles of 128 rows. One CTA per tile (a cluster of n_part CTAs per query)
// when those clusters all fit on the device at once: every CTA then walks one
// tile, the SWA tiles early. Else clusters of min(n_sel, 8) CTAs (one selected
// tile each at k = 512) with the SWA tiles spread over them, when they all fit
// at once: one wave with some CTAs walking two tiles beats two waves. Past one
// wave of those, one CTA per query walks the query's tiles in turn with an
// online softmax (no partials, no merge), as it does whenever the plan comes
// down to one CTA per query. Measured (k = 512, 128 SWA rows,
// L2 flushed): 32 queries 33 us in clusters of 4 against 52 one CTA each; 48
// and 64 queries 60 us in two waves of clusters against 52; 96 queries 89
// against 54; 4,096 prefill queries 2.91 ms in clusters of 5 against 1.38 ms.
// n_q: queries of one launch.
static AttnPlan attn_plan(int32_t n_q, int32_t k, int32_t n_swa, bool query_device) {
  AttnPlan p;
  p.n_sel = (k + attn_tc::kRows - 1) / attn_tc::kRows;
  p.n_swt = (n_swa + attn_tc::kRows - 1) / attn_tc::kRows;
  p.n_part = p.n_sel + p.n_swt;
  int c = p.n_sel < 1 ? 1 : p.n_sel > attn_tc::kMaxCluster ? attn_tc::kMaxCluster : p.n_sel;
  p.seq = false;
  if (query_device) {
    const int fit = p.n_part > c && p.n_part <= attn_tc::kMaxCluster ? attn_max_clusters(p.n_part) : 0;
    if (fit > 0 && fit >= n_q) {
      c = p.n_part;
    } else {
      while (c > 1 && attn_max_clusters(c) < 1) c >>= 1;
      // a cluster of one would only add the merge to the sequential walk
      if (c == 1 || attn_max_clusters(c) < n_q) {
        c = 1;
        p.seq = true;
      }
    }
  }
  p.cluster = c;
  return p;
}

// Reuse mode: a cluster per sequence whose CTAs take the L x n_swt SWA tiles
// and the selected tiles, each selected tile gathered once per group of lgrp
// layers (lgrp = 2 for even L: measured faster than one gather for all L
// layers, whose passes then run back to back on one CTA). Possible when one
// cluster holds the merge of the L x 64 (layer, head) rows: at most 64 rows a
// CTA (C >= L) and the (max, sum) exchange within its shared-memory table.
static bool attn_reuse_plan(int L, AttnPlan& p, int& lgrp) {
  lgrp = L % 2 == 0 ? 2 : L;
  const int items = L * p.n_swt + p.n_sel * (L / lgrp);
  const int c = items < attn_tc::kMaxCluster ? items : attn_tc::kMaxCluster;
  if (c < L) return false;
  const int nh = (kHeads * L + c - 1) / c;
  if (p.n_part * nh > attn_tc::kMaxPartials * 16) return false;
  if (attn_max_clusters(c, true) < 1) return false;
  p.cluster = c;
  return true;
}

static inline int attn_queries_per_launch(int32_t n_queries) {
  return n_queries < kQueriesPerLaunch ? n_queries : kQueriesPerLaunch;
}

static size_t attn_part_o_bytes(int32_t nq, int n_part) {
  size_t o = (size_t)nq * (size_t)n_part * kHeads * kHeadDim * 4;
  return (o + 255) / 256 * 256;
}

extern "C" size_t csa2_sparse_attn_workspace_size(int32_t n_queries, int32_t k, int32_t n_swa) {
  if (n_queries <= 0 || k < 0 || n_swa < 0) return 0;
  // partials are indexed by query within one launch of at most kQueriesPerLaunch
  const int32_t nq = attn_queries_per_launch(n_queries);
  const AttnPlan plan = attn_plan(nq, k, n_swa, false);
  if (plan.n_part == 0) return 256;
  return attn_part_o_bytes(nq, plan.n_part);
}

extern "C" int csa2_sparse_attn_kernel_launches(int32_t n_queries, int32_t k, int32_t n_swa) {
  if (n_queries <= 0 || k < 0 || n_swa < 0) return 0;
  return (n_queries + kQueriesPerLaunch - 1) / kQueriesPerLaunch;
}

static int launch_attn(AttnArgs a, const void* q_bf16, int32_t n_q, uint16_t* out, float* out_f32, float* lse,
                       void* ws, size_t ws_bytes, cudaStream_t stream, bool reuse = false) {
  if (attn_kernel_attr() != CSA2_OK) return CSA2_ERR_CUDA;
  AttnPlan plan = attn_plan(attn_queries_per_launch(n_q), a.k, a.n_swa, true);
  if (plan.n_part > attn_tc::kMaxPartials) return CSA2_ERR_UNSUPPORTED_SHAPE;
  a.n_sel = plan.n_sel;
  a.n_swt = plan.n_swt;
  a.n_part = plan.n_part;
  a.out = out;
  a.out_f32 = out_f32;
  a.lse = lse;
  const size_t need = csa2_sparse_attn_workspace_size(n_q, a.k, a.n_swa);
  if (!ws || ws_bytes < need || !csa2_aligned(ws, 256)) return CSA2_ERR_WORKSPACE;
  a.part_o = (float*)ws;
  // Q rows of all queries as a 2-D bf16 tensor [n_q * 64][512], loaded in
  // [64 heads][64 channels] boxes with the 128-byte swizzle the MMA reads.
  auto encode = tensor_map_encoder();
  if (!encode) return CSA2_ERR_CUDA;
  CUtensorMap qmap;
  cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)n_q * kHeads};
  cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kHeads};
  cuuint32_t estr[2] = {1, 1};
  if (encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q_bf16), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return CSA2_ERR_CUDA;
  int lgrp = 1;
  if (reuse && a.L >= 2) {
    if (!attn_reuse_plan(a.L, plan, lgrp)) return CSA2_ERR_UNSUPPORTED_SHAPE;
    a.lgrp = lgrp;
    // units are sequences: at most kQueriesPerLaunch queries (B x L) a launch
    const int32_t n_seq = n_q / a.L, per = kQueriesPerLaunch / a.L;
    for (int32_t s0 = 0; s0 < n_seq; s0 += per) {
      const int32_t ns = n_seq - s0 < per ? n_seq - s0 : per;
      a.q0 = s0;
      if (csa2_launch_pdl_cluster(attn_tc::attn_tc_kernel<attn_tc::kModeReuse>, dim3((unsigned)plan.cluster, (unsigned)ns),
                                  dim3(attn_tc::kThreads), (size_t)attn_tc::kSmemBytes, stream,
                                  (unsigned)plan.cluster, qmap, a) != cudaSuccess) {
        (void)cudaGetLastError();
        return CSA2_ERR_CUDA;
      }
    }
    return CSA2_OK;
  }
  for (int32_t q0 = 0; q0 < n_q; q0 += kQueriesPerLaunch) {
    const int32_t nq = n_q - q0 < kQueriesPerLaunch ? n_q - q0 : kQueriesPerLaunch;
    a.q0 = q0;
    const auto kern = plan.seq ? attn_tc::attn_tc_kernel<attn_tc::kModeSeq>
                               : attn_tc::attn_tc_kernel<attn_tc::kModeCluster>;
    if (csa2_launch_pdl_cluster(kern, dim3((unsigned)plan.cluster, (unsigned)nq), dim3(attn_tc::kThreads),
                                (size_t)attn_tc::kSmemBytes, stream, (unsigned)plan.cluster, qmap, a) != cudaSuccess) {
      (void)cudaGetLastError();
      return CSA2_ERR_CUDA;
    }
  }
  return CSA2_OK;
}

static int sparse_attn_decode(const void* q_bf16, int32_t B, int32_t L, const uint8_t* kv_data,
                              const uint8_t* kv_scale, int64_t cap, const int32_t* n_visible, const int32_t* idx,
                              int32_t k, const uint8_t* swa, int32_t n_swa, float sm_scale, void* out_bf16,
                              float* out_f32, float* lse, void* workspace, size_t workspace_bytes,
                              csa2_stream_t stream, bool reuse) {
  if (!q_bf16 || !kv_data || !kv_scale || !n_visible || !idx || !out_bf16) return CSA2_ERR_INVALID_ARG;
  if (B < 0 || L < 1 || k < 0 || n_swa < 0 || cap < 0) return CSA2_ERR_INVALID_ARG;
  if (n_swa > 0 && !swa) return CSA2_ERR_INVALID_ARG;
  if (k > CSA2_MAX_TOPK || n_swa > 512) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (!csa2_aligned(q_bf16, 16) || !csa2_aligned(kv_data, 16) || !csa2_aligned(kv_scale, 16) || !csa2_aligned(out_bf16, 8) ||
      (swa && !csa2_aligned(swa, 16)) || (out_f32 && !csa2_aligned(out_f32, 16)))
    return CSA2_ERR_ALIGNMENT;
  if (B == 0) return CSA2_OK;
  AttnArgs a{};
  a.kv_data = kv_data;
  a.kv_scale = kv_scale;
  a.kv_seq_stride = cap;
  a.n_visible = n_visible;
  a.idx = idx;
  a.k = k;
  a.L = L;
  a.lgrp = 1;
  a.swa = swa;
  a.swa_q_stride = (int64_t)n_swa * kHeadDim;
  a.n_swa = n_swa;
  a.swa_first_row = INT32_MIN;  // decode windows are never truncated
  a.sm_scale = sm_scale;
  return launch_attn(a, q_bf16, B * L, (uint16_t*)out_bf16, out_f32, lse, workspace, workspace_bytes,
                     (cudaStream_t)stream, reuse);
}

extern "C" int csa2_sparse_attn_decode(const void* q_bf16, int32_t B, int32_t L, const uint8_t* kv_data,
                                       const uint8_t* kv_scale, int64_t cap, const int32_t* n_visible,
                                       const int32_t* idx, int32_t k, const uint8_t* swa, int32_t n_swa,
                                       float sm_scale, void* out_bf16, float* out_f32, float* lse, void* workspace,
                                       size_t workspace_bytes, csa2_stream_t stream) {
  return sparse_attn_decode(q_bf16, B, L, kv_data, kv_scale, cap, n_visible, idx, k, swa, n_swa, sm_scale, out_bf16,
                            out_f32, lse, workspace, workspace_bytes, stream, false);
}

extern "C" int csa2_sparse_attn_reuse(const void* q_bf16, int32_t B, int32_t L, const uint8_t* kv_data,
                                      const uint8_t* kv_scale, int64_t cap, const int32_t* n_visible,
                                      const int32_t* idx, int32_t k, const uint8_t* swa, int32_t n_swa,
                                      float sm_scale, void* out_bf16, float* out_f32, float* lse, void* workspace,
                                      size_t workspace_bytes, csa2_stream_t stream) {
  return sparse_attn_decode(q_bf16, B, L, kv_data, kv_scale, cap, n_visible, idx, k, swa, n_swa, sm_scale, out_bf16,
                            out_f32, lse, workspace, workspace_bytes, stream, true);
}

extern "C" int csa2_sparse_attn_prefill_replay(const void* q_bf16, int32_t T, const uint8_t* kv_data,
                                               const uint8_t* kv_scale, int64_t n_entries, const int32_t* idx,
                                               int32_t k, const uint8_t* swa, int32_t n_swa, int32_t replay_row,
                                               float sm_scale, void* out_bf16, float* out_f32, float* lse,
                                               void* workspace, size_t workspace_bytes, csa2_stream_t stream) {
  if (!q_bf16 || !kv_data || !kv_scale || !idx || !out_bf16) return CSA2_ERR_INVALID_ARG;
  if (T < 0 || k < 0 || n_swa < 0 || n_entries < 0 || replay_row < 0) return CSA2_ERR_INVALID_ARG;
  if (n_swa > 0 && !swa) return CSA2_ERR_INVALID_ARG;
  if (k > CSA2_MAX_TOPK || n_swa > 512) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (!csa2_aligned(q_bf16, 16) || !csa2_aligned(kv_data, 16) || !csa2_aligned(kv_scale, 16) || !csa2_aligned(out_bf16, 8) ||
      (swa && !csa2_aligned(swa, 16)) || (out_f32 && !csa2_aligned(out_f32, 16)))
    return CSA2_ERR_ALIGNMENT;
  if (T == 0) return CSA2_OK;
  AttnArgs a{};
  a.kv_data = kv_data;
  a.kv_scale = kv_scale;
  a.kv_seq_stride = 0;
  a.n_visible = nullptr;
  a.nv_const = n_entries;
  a.idx = idx;
  a.k = k;
  a.L = 1;
  a.lgrp = 1;
  a.swa = swa;
  a.swa_q_stride = kHeadDim;  // query t uses rows t .. t + n_swa - 1
  a.n_swa = n_swa;
  a.swa_first_row = replay_row;
  a.sm_scale = sm_scale;
  return launch_attn(a, q_bf16, T, (uint16_t*)out_bf16, out_f32, lse, workspace, workspace_bytes, (cudaStream_t)stream);
}

extern "C" int csa2_sparse_attn_prefill(const void* q_bf16, int32_t T, const uint8_t* kv_data,
                                        const uint8_t* kv_scale, int64_t n_entries, const int32_t* idx, int32_t k,
                                        const uint8_t* swa, int32_t n_swa, float sm_scale, void* out_bf16,
                                        float* out_f32, float* lse, void* workspace, size_t workspace_bytes,
                                        csa2_stream_t stream) {
  return csa2_sparse_attn_prefill_replay(q_bf16, T, kv_data, kv_scale, n_entries, idx, k, swa, n_swa, 0, sm_scale,
                                         out_bf16, out_f32, lse, workspace, workspace_bytes, stream);
}
