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
// Work split: one CTA per (query, chunk of kRows rows) computes an
// unnormalised partial (m, l, O) of its rows; a second kernel merges the
// chunks of a query in fixed chunk order, so results are deterministic.
#include "common.cuh"

namespace csa2 {

__device__ int g_attn_error = 0;

constexpr int kRows = 64;                 // rows (selected entries or SWA rows) per CTA
constexpr int kThreads = 256;
constexpr int kQStride = kHeadDim + 8;    // bf16 elements per smem row (padded)
constexpr int kSStride = kRows + 1;

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
  float sm_scale;
  int32_t n_split;
  float* part_o;            // [n_q][n_split][64][512]
  float* part_ml;           // [n_q][n_split][64][2]
  int32_t q0;               // first query of this launch
};

__device__ __forceinline__ void dequant_kv_block16(const uint8_t* d8, uint8_t s8, uint16_t* dst) {
  uint2 v = *reinterpret_cast<const uint2*>(d8);
  float s = e4m3_to_f32(s8);
  uint32_t w[2] = {v.x, v.y};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t b = (w[i] >> (8 * j)) & 0xFFu;
      __nv_bfloat162 p = __floats2bfloat162_rn(e2m1_to_f32(b & 0xF) * s, e2m1_to_f32(b >> 4) * s);
      o[4 * i + j] = *reinterpret_cast<uint32_t*>(&p);
    }
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(o[0], o[1], o[2], o[3]);
  d[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ void dequant_swa16(const uint8_t* src, uint16_t* dst) {
  uint4 v = *reinterpret_cast<const uint4*>(src);
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t b = w[i] >> (16 * j);
      __nv_bfloat162 p = __floats2bfloat162_rn(e4m3_to_f32(b & 0xFF), e4m3_to_f32((b >> 8) & 0xFF));
      o[2 * i + j] = *reinterpret_cast<uint32_t*>(&p);
    }
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(o[0], o[1], o[2], o[3]);
  d[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ void bf16x8_to_f32(uint4 v, float* f) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// grid (n_split, n_q_in_launch), block kThreads
__global__ void __launch_bounds__(kThreads) attn_partial_kernel(AttnArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem);                    // [64][kQStride]
  uint16_t* KVs = Qs + kHeads * kQStride;                             // [kRows][kQStride]
  float* Ss = reinterpret_cast<float*>(KVs + kRows * kQStride);        // [64][kSStride]
  __shared__ int row_valid[kRows];
  __shared__ float m_s[kHeads], l_s[kHeads];

  const int qi = a.q0 + blockIdx.y;            // global query index
  const int seq = qi / a.L;
  const int split = blockIdx.x;
  const int tid = threadIdx.x;

  // ---- load Q (64 x 512 bf16) ----
  const uint16_t* qg = a.q + (int64_t)qi * kHeads * kHeadDim;
  for (int i = tid; i < kHeads * kHeadDim / 8; i += kThreads) {
    int h = i / (kHeadDim / 8), c8 = i % (kHeadDim / 8);
    *reinterpret_cast<uint4*>(Qs + h * kQStride + c8 * 8) =
        *reinterpret_cast<const uint4*>(qg + h * kHeadDim + c8 * 8);
  }
  // ---- gather + dequantise the chunk's rows ----
  const int64_t nv = a.n_visible ? (int64_t)a.n_visible[seq] : a.nv_const;
  const int32_t* idx_row = a.idx + (int64_t)seq * a.k;
  if (tid < kRows) {
    int t = split * kRows + tid;
    int valid = 0;
    if (t < a.k) {
      int32_t p = idx_row[t];
      if (p >= 0) {
        if (p < nv) valid = 1;
        else record_error(&g_attn_error, CSA2_ERR_DEVICE);
      }
    } else if (t < a.k + a.n_swa) {
      valid = 1;
    }
    row_valid[tid] = valid;
  }
  __syncthreads();
  for (int i = tid; i < kRows * (kHeadDim / 16); i += kThreads) {
    int r = i / (kHeadDim / 16), blk = i % (kHeadDim / 16);
    int t = split * kRows + r;
    uint16_t* dst = KVs + r * kQStride + blk * 16;
    if (!row_valid[r]) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(dst + 8) = make_uint4(0, 0, 0, 0);
    } else if (t < a.k) {
      int64_t p = (int64_t)seq * a.kv_seq_stride + idx_row[t];
      dequant_kv_block16(a.kv_data + p * kKvBytes + blk * 8, a.kv_scale[p * kKvScales + blk], dst);
    } else {
      const uint8_t* src = a.swa + (int64_t)qi * a.swa_q_stride + (int64_t)(t - a.k) * kHeadDim + blk * 16;
      dequant_swa16(src, dst);
    }
  }
  __syncthreads();

  // ---- S = sm_scale * Q . KV^T over the chunk: thread owns 4 heads x 4 rows ----
  {
    const int h0 = (tid >> 4) * 4, r0 = (tid & 15) * 4;
    float acc[4][4] = {};
    for (int c = 0; c < kHeadDim; c += 8) {
      float qf[4][8], kf[4][8];
#pragma unroll
      for (int i = 0; i < 4; ++i) bf16x8_to_f32(*reinterpret_cast<const uint4*>(Qs + (h0 + i) * kQStride + c), qf[i]);
#pragma unroll
      for (int j = 0; j < 4; ++j) bf16x8_to_f32(*reinterpret_cast<const uint4*>(KVs + (r0 + j) * kQStride + c), kf[j]);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[i][j] = fmaf(qf[i][e], kf[j][e], acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        Ss[(h0 + i) * kSStride + r0 + j] = row_valid[r0 + j] ? acc[i][j] * a.sm_scale : -INFINITY;
  }
  __syncthreads();

  // ---- per-head max / exp / sum over the chunk: one warp per 8 heads ----
  {
    const int warp = tid >> 5, lane = tid & 31;
    for (int h = warp * 8; h < warp * 8 + 8; ++h) {
      float s0 = Ss[h * kSStride + lane], s1 = Ss[h * kSStride + lane + 32];
      float m = fmaxf(s0, s1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float p0 = (s0 == -INFINITY) ? 0.0f : expf(s0 - m);
      float p1 = (s1 == -INFINITY) ? 0.0f : expf(s1 - m);
      float l = p0 + p1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      Ss[h * kSStride + lane] = p0;
      Ss[h * kSStride + lane + 32] = p1;
      if (lane == 0) { m_s[h] = m; l_s[h] = l; }
    }
  }
  __syncthreads();

  // ---- O_partial = P . KV: warp owns 4 heads, lane owns 16 channels; 2 passes ----
  const int lq = blockIdx.y;                  // query within this launch
  float* po = a.part_o + ((int64_t)lq * a.n_split + split) * kHeads * kHeadDim;
  {
    const int warp = tid >> 5, lane = tid & 31;
    const int c0 = lane * 16;
    for (int pass = 0; pass < 2; ++pass) {
      const int h0 = pass * 32 + warp * 4;
      float acc[4][16] = {};
      for (int r = 0; r < kRows; ++r) {
        float kf[16];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(KVs + r * kQStride + c0), kf);
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(KVs + r * kQStride + c0 + 8), kf + 8);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float p = Ss[(h0 + i) * kSStride + r];
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[i][e] = fmaf(p, kf[e], acc[i][e]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float4* d = reinterpret_cast<float4*>(po + (h0 + i) * kHeadDim + c0);
#pragma unroll
        for (int e = 0; e < 4; ++e) d[e] = make_float4(acc[i][4 * e], acc[i][4 * e + 1], acc[i][4 * e + 2], acc[i][4 * e + 3]);
      }
    }
  }
  if (tid < kHeads) {
    float* ml = a.part_ml + (((int64_t)lq * a.n_split + split) * kHeads + tid) * 2;
    ml[0] = m_s[tid];
    ml[1] = l_s[tid];
  }
}

// grid (n_q_in_launch), block 256: merge the splits of each (query, head) in
// fixed split order.
__global__ void __launch_bounds__(256) attn_combine_kernel(const float* __restrict__ part_o,
                                                           const float* __restrict__ part_ml, int32_t n_split,
                                                           int32_t q0, uint16_t* __restrict__ out,
                                                           float* __restrict__ out_f32, float* __restrict__ lse) {
  __shared__ float scale_s[kHeads][16];
  __shared__ float inv_l[kHeads];
  const int lq = blockIdx.x;
  const int qi = q0 + lq;
  const int tid = threadIdx.x;
  if (tid < kHeads) {
    float M = -INFINITY;
    for (int s = 0; s < n_split; ++s) {
      const float* ml = part_ml + (((int64_t)lq * n_split + s) * kHeads + tid) * 2;
      if (ml[1] > 0.0f) M = fmaxf(M, ml[0]);
    }
    float Lsum = 0.0f;
    for (int s = 0; s < n_split; ++s) {
      const float* ml = part_ml + (((int64_t)lq * n_split + s) * kHeads + tid) * 2;
      float f = (ml[1] > 0.0f) ? expf(ml[0] - M) : 0.0f;
      scale_s[tid][s] = f;
      Lsum += ml[1] * f;
    }
    inv_l[tid] = Lsum > 0.0f ? 1.0f / Lsum : 0.0f;
    if (lse) lse[(int64_t)qi * kHeads + tid] = Lsum > 0.0f ? M + logf(Lsum) : -INFINITY;
  }
  __syncthreads();
  for (int i = tid; i < kHeads * kHeadDim / 4; i += blockDim.x) {
    int h = i / (kHeadDim / 4), c4 = i % (kHeadDim / 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < n_split; ++s) {
      float f = scale_s[h][s];
      if (f == 0.0f) continue;
      float4 v = *reinterpret_cast<const float4*>(part_o + (((int64_t)lq * n_split + s) * kHeads + h) * kHeadDim + c4 * 4);
      acc.x = fmaf(v.x, f, acc.x); acc.y = fmaf(v.y, f, acc.y);
      acc.z = fmaf(v.z, f, acc.z); acc.w = fmaf(v.w, f, acc.w);
    }
    float il = inv_l[h];
    acc.x *= il; acc.y *= il; acc.z *= il; acc.w *= il;
    int64_t o = ((int64_t)qi * kHeads + h) * kHeadDim + c4 * 4;
    if (out_f32) *reinterpret_cast<float4*>(out_f32 + o) = acc;
    __nv_bfloat162 b0 = __floats2bfloat162_rn(acc.x, acc.y), b1 = __floats2bfloat162_rn(acc.z, acc.w);
    *reinterpret_cast<uint2*>(out + o) = make_uint2(*reinterpret_cast<uint32_t*>(&b0), *reinterpret_cast<uint32_t*>(&b1));
  }
}

}  // namespace csa2

using namespace csa2;

static constexpr int kMaxSplit = 16;  // k + n_swa <= 1024 rows per query
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

static inline int attn_splits(int32_t k, int32_t n_swa) { return (k + n_swa + kRows - 1) / kRows; }

static inline size_t attn_smem_bytes() {
  return (size_t)(kHeads + kRows) * kQStride * 2 + (size_t)kHeads * kSStride * 4;
}

extern "C" size_t csa2_sparse_attn_workspace_size(int32_t n_queries, int32_t k, int32_t n_swa) {
  if (n_queries <= 0 || k < 0 || n_swa < 0) return 0;
  // partials are indexed by query within one launch of at most kQueriesPerLaunch
  int32_t nq = n_queries < kQueriesPerLaunch ? n_queries : kQueriesPerLaunch;
  int ns = attn_splits(k, n_swa);
  if (ns < 1) ns = 1;
  size_t o = (size_t)nq * ns * kHeads * kHeadDim * 4;
  o = (o + 255) / 256 * 256;
  return o + (size_t)nq * ns * kHeads * 2 * 4;
}

static int launch_attn(AttnArgs a, int32_t n_q, uint16_t* out, float* out_f32, float* lse, void* ws, size_t ws_bytes,
                       cudaStream_t stream) {
  a.n_split = attn_splits(a.k, a.n_swa);
  if (a.n_split < 1) a.n_split = 1;
  if (a.n_split > kMaxSplit) return CSA2_ERR_UNSUPPORTED_SHAPE;
  size_t need = csa2_sparse_attn_workspace_size(n_q, a.k, a.n_swa);
  if (!ws || ws_bytes < need || !csa2_aligned(ws, 256)) return CSA2_ERR_WORKSPACE;
  int32_t nq_ws = n_q < kQueriesPerLaunch ? n_q : kQueriesPerLaunch;
  size_t o_bytes = (size_t)nq_ws * a.n_split * kHeads * kHeadDim * 4;
  o_bytes = (o_bytes + 255) / 256 * 256;
  a.part_o = (float*)ws;
  a.part_ml = (float*)((char*)ws + o_bytes);
  size_t smem = attn_smem_bytes();
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(attn_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return CSA2_ERR_CUDA;
    attr = true;
  }
  for (int32_t q0 = 0; q0 < n_q; q0 += kQueriesPerLaunch) {
    int32_t nq = n_q - q0 < kQueriesPerLaunch ? n_q - q0 : kQueriesPerLaunch;
    a.q0 = q0;
    attn_partial_kernel<<<dim3((unsigned)a.n_split, (unsigned)nq), kThreads, smem, stream>>>(a);
    CSA2_CHECK_LAUNCH();
    attn_combine_kernel<<<(unsigned)nq, 256, 0, stream>>>(a.part_o, a.part_ml, a.n_split, q0, out, out_f32, lse);
    CSA2_CHECK_LAUNCH();
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
  if (k > CSA2_MAX_TOPK || n_swa > 512 || attn_splits(k, n_swa) > kMaxSplit) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (!csa2_aligned(q_bf16, 16) || !csa2_aligned(kv_data, 8) || !csa2_aligned(out_bf16, 8) ||
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
  a.sm_scale = sm_scale;
  return launch_attn(a, B * L, (uint16_t*)out_bf16, out_f32, lse, workspace, workspace_bytes, (cudaStream_t)stream);
}

extern "C" int csa2_sparse_attn_prefill(const void* q_bf16, int32_t T, const uint8_t* kv_data,
                                        const uint8_t* kv_scale, int64_t n_entries, const int32_t* idx, int32_t k,
                                        const uint8_t* swa, int32_t n_swa, float sm_scale, void* out_bf16,
                                        float* out_f32, float* lse, void* workspace, size_t workspace_bytes,
                                        csa2_stream_t stream) {
  if (!q_bf16 || !kv_data || !kv_scale || !idx || !out_bf16) return CSA2_ERR_INVALID_ARG;
  if (T < 0 || k < 0 || n_swa < 0 || n_entries < 0) return CSA2_ERR_INVALID_ARG;
  if (n_swa > 0 && !swa) return CSA2_ERR_INVALID_ARG;
  if (k > CSA2_MAX_TOPK || n_swa > 512 || attn_splits(k, n_swa) > kMaxSplit) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (!csa2_aligned(q_bf16, 16) || !csa2_aligned(kv_data, 8) || !csa2_aligned(out_bf16, 8) ||
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
  a.sm_scale = sm_scale;
  return launch_attn(a, T, (uint16_t*)out_bf16, out_f32, lse, workspace, workspace_bytes, (cudaStream_t)stream);
}
