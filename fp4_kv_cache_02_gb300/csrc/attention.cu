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
// Work split: one CTA per (query, chunk of rows) computes an unnormalised
// partial (m, l, O) of its rows on the tensor cores (attention_tc.cuh); a
// second kernel merges the chunks of a query in fixed chunk order, so results
// are deterministic. The chunk size (32 .. 160 rows) is picked per launch so
// that the CTAs fill the SMs in as few waves as possible.
#include <cooperative_groups.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace csa2 {

__device__ int g_attn_error = 0;

struct AttnArgs {
  const uint16_t* q;        // query rows, [n_q][64][512] bf16
  const uint8_t* kv_data;   // plane base
  const uint8_t* kv_scale;
  int64_t kv_seq_stride;    // entries between sequences (0: one shared plane)
  const int32_t* n_visible; // per sequence, or null (then nv_const)
  int64_t nv_const;
  const int32_t* idx;       // [n_seq][k]
  int32_t k;
  int32_t L;                // queries per sequence (layers sharing the Top-K)
  const uint8_t* swa;       // SWA bytes
  int64_t swa_q_stride;     // bytes between consecutive queries' windows
  int32_t n_swa;
  int32_t swa_first_row;    // prefill: SWA rows before this row of the array are masked (Bounded Replay)
  float sm_scale;
  int32_t n_split;
  int32_t rows;             // rows per chunk (a multiple of 32, at most 160)
  float* part_o;            // [n_q][n_split][64][512]
  float* part_ml;           // [n_q][n_split][64][2]
  int32_t q0;               // first query of this launch
  int32_t fused;            // the n_split CTAs of a query form a cluster and merge in shared memory
  uint16_t* out;            // [n_q][64][512] bf16 (fused path)
  float* out_f32;           // nullable (fused path)
  float* lse;               // nullable (fused path)
};

constexpr int kMaxSplitCombine = 32;

// grid (n_q_in_launch, 8), block 512: merge the splits of 8 heads of one
// query, in fixed split order. Thread t owns the float4 columns t and t + 512
// of the CTA's [8 heads][512] output; it issues the loads of its first batch of
// splits before the (max, sum) of the splits are read and turned into weights.
constexpr int kCombineThreads = 512;
__global__ void __launch_bounds__(kCombineThreads) attn_combine_kernel(const float* __restrict__ part_o,
                                                                       const float* __restrict__ part_ml,
                                                                       int32_t n_split, int32_t q0,
                                                                       uint16_t* __restrict__ out,
                                                                       float* __restrict__ out_f32,
                                                                       float* __restrict__ lse) {
  pdl_begin();
  constexpr int kHeadsPerCta = 8;
  constexpr int kBatch = 8;                      // splits loaded together
  constexpr int kItems = kHeadsPerCta * kHeadDim / 4 / kCombineThreads;  // 2 float4 per thread
  __shared__ float ml_s[kMaxSplitCombine][kHeadsPerCta][2];
  __shared__ float scale_s[kHeadsPerCta][kMaxSplitCombine];
  __shared__ float inv_l[kHeadsPerCta];
  const int lq = blockIdx.x;
  const int qi = q0 + lq;
  const int h0 = blockIdx.y * kHeadsPerCta;
  const int tid = threadIdx.x;
  const int64_t split_stride = (int64_t)kHeads * kHeadDim;
  const float* qbase = part_o + (int64_t)lq * n_split * split_stride + (int64_t)h0 * kHeadDim;
  float4 v[kItems][kBatch];
  auto load_batch = [&](int s0) {
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      const int i = tid + u * kCombineThreads;  // [hl][c4] within the CTA's heads
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        v[u][j] = s0 + j < n_split ? *reinterpret_cast<const float4*>(qbase + (s0 + j) * split_stride + i * 4)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  load_batch(0);
  if (tid < n_split * kHeadsPerCta) {
    const int sp = tid / kHeadsPerCta, hl = tid % kHeadsPerCta;
    const float2 ml = *reinterpret_cast<const float2*>(part_ml + (((int64_t)lq * n_split + sp) * kHeads + h0 + hl) * 2);
    ml_s[sp][hl][0] = ml.x;
    ml_s[sp][hl][1] = ml.y;
  }
  __syncthreads();
  if (tid < kHeadsPerCta) {
    float M = -INFINITY;
    for (int sp = 0; sp < n_split; ++sp)
      if (ml_s[sp][tid][1] > 0.0f) M = fmaxf(M, ml_s[sp][tid][0]);
    float Lsum = 0.0f;
    for (int sp = 0; sp < n_split; ++sp) {
      const float f = ml_s[sp][tid][1] > 0.0f ? expf(ml_s[sp][tid][0] - M) : 0.0f;
      scale_s[tid][sp] = f;
      Lsum += ml_s[sp][tid][1] * f;
    }
    inv_l[tid] = Lsum > 0.0f ? 1.0f / Lsum : 0.0f;
    if (lse) lse[(int64_t)qi * kHeads + h0 + tid] = Lsum > 0.0f ? M + logf(Lsum) : -INFINITY;
  }
  __syncthreads();
  float4 acc[kItems];
#pragma unroll
  for (int u = 0; u < kItems; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < n_split; s0 += kBatch) {
    if (s0 > 0) load_batch(s0);
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      const int hl = (tid + u * kCombineThreads) / (kHeadDim / 4);
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (s0 + j >= n_split) break;
        const float f = scale_s[hl][s0 + j];  // fixed split order
        acc[u].x = fmaf(v[u][j].x, f, acc[u].x);
        acc[u].y = fmaf(v[u][j].y, f, acc[u].y);
        acc[u].z = fmaf(v[u][j].z, f, acc[u].z);
        acc[u].w = fmaf(v[u][j].w, f, acc[u].w);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kItems; ++u) {
    const int i = tid + u * kCombineThreads;
    const int hl = i / (kHeadDim / 4), c4 = i % (kHeadDim / 4);
    const float il = inv_l[hl];
    float4 r = acc[u];
    r.x *= il; r.y *= il; r.z *= il; r.w *= il;
    const int64_t o = ((int64_t)qi * kHeads + h0 + hl) * kHeadDim + c4 * 4;
    if (out_f32) *reinterpret_cast<float4*>(out_f32 + o) = r;
    const __nv_bfloat162 b0 = __floats2bfloat162_rn(r.x, r.y), b1 = __floats2bfloat162_rn(r.z, r.w);
    *reinterpret_cast<uint2*>(out + o) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1));
  }
}

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

static constexpr int kMaxSplit = kMaxSplitCombine;  // k + n_swa <= 32 x 160 rows per query
static constexpr int kQueriesPerLaunch = 256;

int csa2_read_and_clear_attn_error(cudaStream_t s) {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_attn_error, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return CSA2_ERR_CUDA;
  if (cudaMemcpyToSymbolAsync(g_attn_error, &z, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return CSA2_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return CSA2_ERR_CUDA;
  return v;
}

static int sm_count() {
  constexpr int kMaxDevices = 64;
  static int count[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
  if (!count[dev]) {
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) c = 152;
    count[dev] = c;
  }
  return count[dev];
}

static constexpr int kMaxClusterSplit = attn_tc::kMaxClusterChunks;  // portable cluster size

// Opts the partial kernel into its dynamic shared memory, once per device.
static int attn_kernel_attr() {
  static Csa2PerDeviceOnce optin;
  return csa2_smem_optin((const void*)attn_tc::attn_partial_tc_kernel, attn_tc::kSmemBytes, optin);
}

// How many clusters of `size` partial CTAs can be resident at once (0 when a
// cluster of that size cannot run), cached per device.
static int attn_max_clusters(int size) {
  constexpr int kMaxDevices = 64;
  static int cache[kMaxDevices][kMaxClusterSplit + 1];
  static bool filled[kMaxDevices][kMaxClusterSplit + 1];
  int dev = 0;
  if (size < 1 || size > kMaxClusterSplit) return 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (!filled[dev][size]) {
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
      if (cudaOccupancyMaxActiveClusters(&n, (void*)attn_tc::attn_partial_tc_kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
      }
    }
    cache[dev][size] = n;
    filled[dev][size] = true;
  }
  return cache[dev][size];
}

struct AttnPlan {
  int rows;    // rows per chunk
  int splits;  // chunks per query
  bool fused;  // chunks of a query form a cluster and merge in shared memory
};

// The chunking of n_q queries of `total` rows each: rows per chunk a multiple
// of 32 (at most 160), merged either inside a cluster (at most 8 chunks) or by
// the combine kernel, whichever has the smaller estimated time = waves x
// (fixed + per-row cost) + merge cost. The costs are the kernels' measured
// times on GB300: about 7.5 us per CTA plus 0.047 us per row; the cluster
// merge about 2.5 us plus 0.6 us per chunk (it waits for the slowest chunk of
// the cluster); the combine kernel about 6 us plus 0.05 us per chunk.
static AttnPlan attn_plan(int32_t n_q, int32_t total) {
  AttnPlan best_plan{-1, 0, false};
  if (total <= 0) return AttnPlan{32, 1, false};
  const int n_sm = sm_count();
  double best = 1e300;
  for (int rows = 32; rows <= attn_tc::kMaxRows; rows += 32) {
    const int splits = (total + rows - 1) / rows;
    if (splits > kMaxSplit) continue;
    const double cta = 7.5 + 0.047 * rows;
    const int64_t waves = ((int64_t)n_q * splits + n_sm - 1) / n_sm;
    const double t = (double)waves * cta + 6.0 + 0.05 * splits;
    if (t < best - 1e-9) {
      best = t;
      best_plan = AttnPlan{rows, splits, false};
    }
    const int clusters = splits <= kMaxClusterSplit ? attn_max_clusters(splits) : 0;
    if (clusters > 0) {
      const int64_t cwaves = ((int64_t)n_q + clusters - 1) / clusters;
      const double tc_ = (double)cwaves * (cta + 2.5 + 0.6 * splits);
      if (tc_ < best - 1e-9) {
        best = tc_;
        best_plan = AttnPlan{rows, splits, true};
      }
    }
  }
  return best_plan;
}

static inline int attn_queries_per_launch(int32_t n_queries) {
  return n_queries < kQueriesPerLaunch ? n_queries : kQueriesPerLaunch;
}

static inline AttnPlan attn_plan_for(int32_t n_queries, int32_t k, int32_t n_swa) {
  return attn_plan(attn_queries_per_launch(n_queries), k + n_swa);
}

extern "C" size_t csa2_sparse_attn_workspace_size(int32_t n_queries, int32_t k, int32_t n_swa) {
  if (n_queries <= 0 || k < 0 || n_swa < 0) return 0;
  // partials are indexed by query within one launch of at most kQueriesPerLaunch
  int32_t nq = attn_queries_per_launch(n_queries);
  const AttnPlan plan = attn_plan_for(n_queries, k, n_swa);
  if (plan.fused) return 256;  // the chunks merge in shared memory
  int ns = plan.splits < 1 ? 1 : plan.splits;
  size_t o = (size_t)nq * ns * kHeads * kHeadDim * 4;
  o = (o + 255) / 256 * 256;
  return o + (size_t)nq * ns * kHeads * 2 * 4;
}

extern "C" int csa2_sparse_attn_kernel_launches(int32_t n_queries, int32_t k, int32_t n_swa) {
  if (n_queries <= 0 || k < 0 || n_swa < 0) return 0;
  const AttnPlan plan = attn_plan_for(n_queries, k, n_swa);
  if (plan.rows < 0) return 0;
  const int batches = (n_queries + kQueriesPerLaunch - 1) / kQueriesPerLaunch;
  return batches * (plan.fused ? 1 : 2);
}

static int launch_attn(AttnArgs a, int32_t n_q, uint16_t* out, float* out_f32, float* lse, void* ws, size_t ws_bytes,
                       cudaStream_t stream) {
  const AttnPlan plan = attn_plan_for(n_q, a.k, a.n_swa);
  if (plan.rows < 0 || plan.splits < 1 || plan.splits > kMaxSplit) return CSA2_ERR_UNSUPPORTED_SHAPE;
  a.n_split = plan.splits;
  a.rows = plan.rows;
  a.fused = plan.fused ? 1 : 0;
  a.out = out;
  a.out_f32 = out_f32;
  a.lse = lse;
  size_t need = csa2_sparse_attn_workspace_size(n_q, a.k, a.n_swa);
  if (!ws || ws_bytes < need || !csa2_aligned(ws, 256)) return CSA2_ERR_WORKSPACE;
  int32_t nq_ws = attn_queries_per_launch(n_q);
  size_t o_bytes = (size_t)nq_ws * a.n_split * kHeads * kHeadDim * 4;
  o_bytes = (o_bytes + 255) / 256 * 256;
  a.part_o = (float*)ws;
  a.part_ml = (float*)((char*)ws + o_bytes);
  if (attn_kernel_attr() != CSA2_OK) return CSA2_ERR_CUDA;
  // Q rows of all queries as a 2-D bf16 tensor [n_q * 64][512], loaded in
  // [64 heads][64 channels] boxes with the 128-byte swizzle the MMA reads.
  auto encode = tensor_map_encoder();
  if (!encode) return CSA2_ERR_CUDA;
  CUtensorMap qmap;
  cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)n_q * kHeads};
  cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kHeads};
  cuuint32_t estr[2] = {1, 1};
  if (encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void*)a.q, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return CSA2_ERR_CUDA;
  for (int32_t q0 = 0; q0 < n_q; q0 += kQueriesPerLaunch) {
    int32_t nq = n_q - q0 < kQueriesPerLaunch ? n_q - q0 : kQueriesPerLaunch;
    a.q0 = q0;
    if (a.fused) {
      if (csa2_launch_pdl_cluster(attn_tc::attn_partial_tc_kernel, dim3((unsigned)a.n_split, (unsigned)nq),
                                  dim3(attn_tc::kThreads), (size_t)attn_tc::kSmemBytes, stream, (unsigned)a.n_split,
                                  qmap, a) != cudaSuccess) {
        (void)cudaGetLastError();
        return CSA2_ERR_CUDA;
      }
    } else {
      CSA2_LAUNCH_PDL(attn_tc::attn_partial_tc_kernel, dim3((unsigned)a.n_split, (unsigned)nq),
                      dim3(attn_tc::kThreads), (size_t)attn_tc::kSmemBytes, stream, qmap, a);
      CSA2_LAUNCH_PDL(attn_combine_kernel, dim3((unsigned)nq, kHeads / 8), dim3(kCombineThreads), 0, stream, a.part_o,
                      a.part_ml, a.n_split, q0, out, out_f32, lse);
    }
  }
  return CSA2_OK;
}

extern "C" int csa2_sparse_attn_decode(const void* q_bf16, int32_t B, int32_t L, const uint8_t* kv_data,
                                       const uint8_t* kv_scale, int64_t cap, const int32_t* n_visible,
                                       const int32_t* idx, int32_t k, const uint8_t* swa, int32_t n_swa,
                                       float sm_scale, void* out_bf16, float* out_f32, float* lse, void* workspace,
                                       size_t workspace_bytes, csa2_stream_t stream) {
  if (!q_bf16 || !kv_data || !kv_scale || !n_visible || !idx || !out_bf16) return CSA2_ERR_INVALID_ARG;
  if (B < 0 || L < 1 || k < 0 || n_swa < 0 || cap < 0) return CSA2_ERR_INVALID_ARG;
  if (n_swa > 0 && !swa) return CSA2_ERR_INVALID_ARG;
  if (k > CSA2_MAX_TOPK || n_swa > 512 || k + n_swa > kMaxSplit * attn_tc::kMaxRows)
    return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (!csa2_aligned(q_bf16, 16) || !csa2_aligned(kv_data, 16) || !csa2_aligned(kv_scale, 2) || !csa2_aligned(out_bf16, 8) ||
      (swa && !csa2_aligned(swa, 16)) || (out_f32 && !csa2_aligned(out_f32, 16)))
    return CSA2_ERR_ALIGNMENT;
  if (B == 0) return CSA2_OK;
  AttnArgs a{};
  a.q = (const uint16_t*)q_bf16;
  a.kv_data = kv_data;
  a.kv_scale = kv_scale;
  a.kv_seq_stride = cap;
  a.n_visible = n_visible;
  a.idx = idx;
  a.k = k;
  a.L = L;
  a.swa = swa;
  a.swa_q_stride = (int64_t)n_swa * kHeadDim;
  a.n_swa = n_swa;
  a.swa_first_row = INT32_MIN;  // decode windows are never truncated
  a.sm_scale = sm_scale;
  return launch_attn(a, B * L, (uint16_t*)out_bf16, out_f32, lse, workspace, workspace_bytes, (cudaStream_t)stream);
}

extern "C" int csa2_sparse_attn_prefill_replay(const void* q_bf16, int32_t T, const uint8_t* kv_data,
                                               const uint8_t* kv_scale, int64_t n_entries, const int32_t* idx,
                                               int32_t k, const uint8_t* swa, int32_t n_swa, int32_t replay_row,
                                               float sm_scale, void* out_bf16, float* out_f32, float* lse,
                                               void* workspace, size_t workspace_bytes, csa2_stream_t stream) {
  if (!q_bf16 || !kv_data || !kv_scale || !idx || !out_bf16) return CSA2_ERR_INVALID_ARG;
  if (T < 0 || k < 0 || n_swa < 0 || n_entries < 0 || replay_row < 0) return CSA2_ERR_INVALID_ARG;
  if (n_swa > 0 && !swa) return CSA2_ERR_INVALID_ARG;
  if (k > CSA2_MAX_TOPK || n_swa > 512 || k + n_swa > kMaxSplit * attn_tc::kMaxRows)
    return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (!csa2_aligned(q_bf16, 16) || !csa2_aligned(kv_data, 16) || !csa2_aligned(kv_scale, 2) || !csa2_aligned(out_bf16, 8) ||
      (swa && !csa2_aligned(swa, 16)) || (out_f32 && !csa2_aligned(out_f32, 16)))
    return CSA2_ERR_ALIGNMENT;
  if (T == 0) return CSA2_OK;
  AttnArgs a{};
  a.q = (const uint16_t*)q_bf16;
  a.kv_data = kv_data;
  a.kv_scale = kv_scale;
  a.kv_seq_stride = 0;
  a.n_visible = nullptr;
  a.nv_const = n_entries;
  a.idx = idx;
  a.k = k;
  a.L = 1;
  a.swa = swa;
  a.swa_q_stride = kHeadDim;  // query t uses rows t .. t + n_swa - 1
  a.n_swa = n_swa;
  a.swa_first_row = replay_row;
  a.sm_scale = sm_scale;
  return launch_attn(a, T, (uint16_t*)out_bf16, out_f32, lse, workspace, workspace_bytes, (cudaStream_t)stream);
}

extern "C" int csa2_sparse_attn_prefill(const void* q_bf16, int32_t T, const uint8_t* kv_data,
                                        const uint8_t* kv_scale, int64_t n_entries, const int32_t* idx, int32_t k,
                                        const uint8_t* swa, int32_t n_swa, float sm_scale, void* out_bf16,
                                        float* out_f32, float* lse, void* workspace, size_t workspace_bytes,
                                        csa2_stream_t stream) {
  return csa2_sparse_attn_prefill_replay(q_bf16, T, kv_data, kv_scale, n_entries, idx, k, swa, n_swa, 0, sm_scale,
                                         out_bf16, out_f32, lse, workspace, workspace_bytes, stream);
}
