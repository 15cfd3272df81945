// shard.cu -- the exchange steps of a decode step split by context across
// ranks: each rank owns the contiguous entries [lo, hi) of every sequence.
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", section
// 2.3 (Top-K over all visible entries; one softmax over the selected rows and
// the SWA window) and section 2.3.2 (the block pool). Splitting the entries
// into ranges keeps every step exact:
//   - a global Top-K winner beats all entries of its own range, so it is in
//     that range's local Top-K: a Top-K over the gathered (score, position)
//     candidates of all ranges reproduces the global one. The same holds for
//     the best blocks of the pool, ranked by their block maxima;
//   - attention over a union of disjoint row sets is the merge of the sets'
//     normalised outputs weighted by exp(lse_r - L), L = log sum_r exp(lse_r).
#include "common.cuh"

namespace csa2 {

// cand[b][j] = (scores[b][c], pos(c) + offset) for the column c = idx[b][j],
// pos(c) = positions[b][c] or c; (-inf, -1) where c or pos(c) is invalid.
__global__ void topk_candidates_kernel(const float* __restrict__ scores, int64_t n, const int32_t* __restrict__ positions,
                                       const int32_t* __restrict__ idx, int32_t k, int64_t offset,
                                       uint2* __restrict__ cand) {
  pdl_begin();
  const int b = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= k) return;
  const int32_t c = idx[(int64_t)b * k + j];
  float v = -INFINITY;
  int32_t p = -1;
  if (c >= 0 && c < n) {
    const int64_t pos = positions ? (int64_t)positions[(int64_t)b * n + c] : (int64_t)c;
    if (pos >= 0) {
      v = scores[(int64_t)b * n + c];
      p = (int32_t)(pos + offset);
    }
  }
  cand[(int64_t)b * k + j] = make_uint2(__float_as_uint(v), (uint32_t)p);
}

// [R][B][k] candidate pairs -> values [B][R*k] and positions [B][R*k]
__global__ void candidates_by_row_kernel(const uint2* __restrict__ cand, int32_t R, int32_t B, int32_t k,
                                         float* __restrict__ vals, int32_t* __restrict__ pos) {
  pdl_begin();
  const int b = blockIdx.y;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t rk = (int64_t)R * k;
  if (i >= rk) return;
  const int r = (int)(i / k), j = (int)(i % k);
  const uint2 c = cand[((int64_t)r * B + b) * k + j];
  vals[(int64_t)b * rk + i] = __uint_as_float(c.x);
  pos[(int64_t)b * rk + i] = (int32_t)c.y;
}

// local[b][j] = idx[b][j] - lo when lo <= idx[b][j] < hi, else -1
__global__ void shard_positions_kernel(const int32_t* __restrict__ idx, int32_t k, int64_t lo, int64_t hi,
                                       int32_t* __restrict__ local) {
  pdl_begin();
  const int b = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= k) return;
  const int32_t p = idx[(int64_t)b * k + j];
  local[(int64_t)b * k + j] = (p >= lo && p < hi) ? (int32_t)(p - lo) : -1;
}

// The positions of the chosen blocks that fall into [lo, hi) and below the
// rank's visible count, as local positions; -1 elsewhere.
__global__ void shard_pool_kernel(const int32_t* __restrict__ blocks, int32_t n_blocks, int32_t block, int64_t lo,
                                  int64_t hi, const int32_t* __restrict__ n_visible, int32_t* __restrict__ pool) {
  pdl_begin();
  const int b = blockIdx.y;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)n_blocks * block) return;
  const int32_t blk = blocks[(int64_t)b * n_blocks + i / block];
  const int64_t nv = n_visible ? (int64_t)n_visible[b] : hi - lo;
  int32_t out = -1;
  if (blk >= 0) {
    const int64_t p = (int64_t)blk * block + i % block;
    if (p >= lo && p < hi && p - lo < nv) out = (int32_t)(p - lo);
  }
  pool[(int64_t)b * n_blocks * block + i] = out;
}

// grid (n_q, 64 heads), 128 threads x 4 channels: merge the R partial outputs
// of one (query, head) in rank order 0..R-1.
__global__ void __launch_bounds__(128) attn_merge_kernel(const float* __restrict__ parts,
                                                         const float* __restrict__ lses, int32_t R, int32_t n_q,
                                                         uint16_t* __restrict__ out, float* __restrict__ out_f32,
                                                         float* __restrict__ lse_out) {
  pdl_begin();
  const int q = blockIdx.x, h = blockIdx.y;
  const int64_t qh = (int64_t)q * kHeads + h;
  const int64_t rstride = (int64_t)n_q * kHeads;
  float L = -INFINITY;
  for (int r = 0; r < R; ++r) L = fmaxf(L, lses[r * rstride + qh]);
  float S = 0.0f;
  if (L != -INFINITY)
    for (int r = 0; r < R; ++r) {
      const float l = lses[r * rstride + qh];
      if (l != -INFINITY) S += expf(l - L);
    }
  const int c = threadIdx.x * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (S > 0.0f) {
    const float inv = 1.0f / S;
    for (int r = 0; r < R; ++r) {
      const float l = lses[r * rstride + qh];
      if (l == -INFINITY) continue;
      const float f = expf(l - L) * inv;
      const float4 v = *reinterpret_cast<const float4*>(parts + (r * rstride + qh) * kHeadDim + c);
      acc.x = fmaf(v.x, f, acc.x);
      acc.y = fmaf(v.y, f, acc.y);
      acc.z = fmaf(v.z, f, acc.z);
      acc.w = fmaf(v.w, f, acc.w);
    }
  }
  const int64_t o = qh * kHeadDim + c;
  if (out_f32) *reinterpret_cast<float4*>(out_f32 + o) = acc;
  const __nv_bfloat162 b0 = __floats2bfloat162_rn(acc.x, acc.y), b1 = __floats2bfloat162_rn(acc.z, acc.w);
  *reinterpret_cast<uint2*>(out + o) =
      make_uint2(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1));
  if (lse_out && threadIdx.x == 0) lse_out[qh] = S > 0.0f ? L + logf(S) : -INFINITY;
}

}  // namespace csa2

using namespace csa2;

int csa2_launch_topk(const float* scores, int32_t B, int64_t n, const int32_t* n_valid, const int32_t* positions,
                     int32_t k, int32_t* idx, void* workspace, size_t workspace_bytes, cudaStream_t stream);

static inline size_t al256(size_t x) { return (x + 255) / 256 * 256; }

extern "C" int csa2_topk_candidates(const float* scores, int32_t B, int64_t n, const int32_t* positions,
                                    const int32_t* idx, int32_t k, int64_t offset, void* cand, csa2_stream_t stream) {
  if (!scores || !idx || !cand || B < 0 || n < 0 || k <= 0 || offset < 0) return CSA2_ERR_INVALID_ARG;
  if (n + offset > 0x7FFFFFFFLL) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (!csa2_aligned(cand, 8)) return CSA2_ERR_ALIGNMENT;
  if (B == 0) return CSA2_OK;
  CSA2_LAUNCH_PDL(topk_candidates_kernel, dim3((unsigned)((k + 255) / 256), (unsigned)B), dim3(256), 0,
                  (cudaStream_t)stream, scores, n, positions, idx, k, offset, (uint2*)cand);
  return CSA2_OK;
}

extern "C" size_t csa2_topk_merge_workspace_size(int32_t R, int32_t B, int32_t k, int32_t k_out) {
  if (R <= 0 || B <= 0 || k <= 0 || k_out <= 0) return 0;
  const int64_t rk = (int64_t)R * k;
  return 2 * al256((size_t)B * rk * 4) + csa2_topk_workspace_size(B, rk, k_out);
}

extern "C" int csa2_topk_merge(const void* cand, int32_t R, int32_t B, int32_t k, int32_t k_out, int32_t* idx,
                               void* workspace, size_t workspace_bytes, csa2_stream_t stream) {
  if (!cand || !idx || R <= 0 || B < 0 || k <= 0) return CSA2_ERR_INVALID_ARG;
  if (k_out <= 0 || k_out > CSA2_MAX_TOPK || (int64_t)R * k > 0x7FFFFFFFLL) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (!csa2_aligned(cand, 8)) return CSA2_ERR_ALIGNMENT;
  if (B == 0) return CSA2_OK;
  const size_t need = csa2_topk_merge_workspace_size(R, B, k, k_out);
  if (!workspace || workspace_bytes < need || !csa2_aligned(workspace, 256)) return CSA2_ERR_WORKSPACE;
  const int64_t rk = (int64_t)R * k;
  char* base = (char*)workspace;
  float* vals = (float*)base;
  int32_t* pos = (int32_t*)(base + al256((size_t)B * rk * 4));
  char* rest = base + 2 * al256((size_t)B * rk * 4);
  cudaStream_t s = (cudaStream_t)stream;
  CSA2_LAUNCH_PDL(candidates_by_row_kernel, dim3((unsigned)((rk + 255) / 256), (unsigned)B), dim3(256), 0, s,
                  (const uint2*)cand, R, B, k, vals, pos);
  return csa2_launch_topk(vals, B, rk, nullptr, pos, k_out, idx, rest, workspace_bytes - (size_t)(rest - base), s);
}

extern "C" int csa2_shard_positions(const int32_t* idx, int32_t B, int32_t k, int64_t lo, int64_t hi,
                                    int32_t* local_idx, csa2_stream_t stream) {
  if (!idx || !local_idx || B < 0 || k <= 0 || lo < 0 || hi < lo) return CSA2_ERR_INVALID_ARG;
  if (B == 0) return CSA2_OK;
  CSA2_LAUNCH_PDL(shard_positions_kernel, dim3((unsigned)((k + 255) / 256), (unsigned)B), dim3(256), 0,
                  (cudaStream_t)stream, idx, k, lo, hi, local_idx);
  return CSA2_OK;
}

extern "C" int csa2_shard_pool(const int32_t* blocks, int32_t B, int32_t n_blocks, int32_t block, int64_t lo,
                               int64_t hi, const int32_t* n_visible, int32_t* pool, csa2_stream_t stream) {
  if (!blocks || !pool || B < 0 || n_blocks <= 0 || block <= 0 || lo < 0 || hi < lo) return CSA2_ERR_INVALID_ARG;
  if ((int64_t)n_blocks * block > 0x7FFFFFFFLL || hi - lo > 0x7FFFFFFFLL) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (B == 0) return CSA2_OK;
  const int64_t total = (int64_t)n_blocks * block;
  CSA2_LAUNCH_PDL(shard_pool_kernel, dim3((unsigned)((total + 255) / 256), (unsigned)B), dim3(256), 0,
                  (cudaStream_t)stream, blocks, n_blocks, block, lo, hi, n_visible, pool);
  return CSA2_OK;
}

extern "C" int csa2_attn_merge(const float* parts, const float* lses, int32_t R, int32_t n_q, void* out_bf16,
                               float* out_f32, float* lse_out, csa2_stream_t stream) {
  if (!parts || !lses || !out_bf16 || R <= 0 || n_q < 0) return CSA2_ERR_INVALID_ARG;
  if (!csa2_aligned(parts, 16) || !csa2_aligned(out_bf16, 8) || (out_f32 && !csa2_aligned(out_f32, 16)))
    return CSA2_ERR_ALIGNMENT;
  if (n_q == 0) return CSA2_OK;
  CSA2_LAUNCH_PDL(attn_merge_kernel, dim3((unsigned)n_q, kHeads), dim3(kHeadDim / 4), 0, (cudaStream_t)stream,
                  parts, lses, R, n_q, (uint16_t*)out_bf16, out_f32, lse_out);
  return CSA2_OK;
}
