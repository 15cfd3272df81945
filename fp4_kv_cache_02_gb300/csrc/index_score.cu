// index_score.cu -- lightning-indexer scores over the MXFP4 indexer-K planes.
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", section
// 2.3 (indexer scores main-KV entries with indexer Q and indexer K), 2.3.1
// (Full and Reindex layers run the indexer) and 2.3.2 (Reindex layers score
// only the candidate pool); mer.dev notes section 4.4 (32 x 128 multiply-adds
// per query-entry pair, ReLU-weighted sum over heads).
//
//   s[b][i] = sum_h w[b][h] * ReLU( qhat[b][h] . khat[b][p_i] )
//
// The decode scan (contiguous entries, or a positions list for Reindex
// layers) runs on the tensor cores (index_score_tc.cuh); the CUDA-core
// kernel here serves the prefill scan.
#include "common.cuh"

namespace csa2 {

__device__ int g_index_error = 0;

}  // namespace csa2

#include "index_score_tc.cuh"

namespace csa2 {

// Dequantise one query's MXFP4 q into shared memory [32][128] fp32.
__device__ __forceinline__ void load_qhat(const uint8_t* __restrict__ q_data,
                                          const uint8_t* __restrict__ q_e8m0, float* qs) {
  for (int i = threadIdx.x; i < kIdxHeads * kIdxDim; i += blockDim.x) {
    int h = i / kIdxDim, c = i % kIdxDim;
    uint32_t byte = q_data[h * kIkBytes + c / 2];
    uint32_t code = (c & 1) ? (byte >> 4) : (byte & 0xF);
    qs[i] = e2m1_to_f32(code) * e8m0_to_f32(q_e8m0[h * kIkScales + c / 32]);
  }
}

// Score of one key row against the shared qhat: per 32-channel block the key
// values are decoded into registers and folded into 32 per-head partial dots.
__device__ __forceinline__ float score_row(const uint8_t* __restrict__ kd,
                                           const uint8_t* __restrict__ ksc,
                                           const float* qs, const float* ws) {
  float dot[kIdxHeads];
#pragma unroll
  for (int h = 0; h < kIdxHeads; ++h) dot[h] = 0.0f;
  uint32_t scales = *reinterpret_cast<const uint32_t*>(ksc);
#pragma unroll 1
  for (int kb = 0; kb < 4; ++kb) {
    uint4 v = *reinterpret_cast<const uint4*>(kd + kb * 16);
    float s = e8m0_to_f32((scales >> (8 * kb)) & 0xFF);
    uint32_t words[4] = {v.x, v.y, v.z, v.w};
    float kv[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) kv[i] = e2m1_to_f32((words[i / 8] >> (4 * (i % 8))) & 0xF) * s;
#pragma unroll
    for (int h = 0; h < kIdxHeads; ++h) {
      const float* qrow = qs + h * kIdxDim + kb * 32;
      float acc = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) acc = fmaf(qrow[i], kv[i], acc);
      dot[h] += acc;
    }
  }
  float s = 0.0f;
#pragma unroll
  for (int h = 0; h < kIdxHeads; ++h) s = fmaf(ws[h], fmaxf(dot[h], 0.0f), s);
  return s;
}

// Prefill: grid (ceil(n_entries / blockDim), T); query t sees 0..p0+t.
__global__ void __launch_bounds__(128) prefill_score_simple_kernel(
    const uint8_t* __restrict__ q_data, const uint8_t* __restrict__ q_e8m0,
    const float* __restrict__ w, const uint8_t* __restrict__ ik_data,
    const uint8_t* __restrict__ ik_scale, int64_t n_entries, int64_t p0,
    float* __restrict__ scores) {
  __shared__ float qs[kIdxHeads * kIdxDim];
  __shared__ float ws[kIdxHeads];
  const int t = blockIdx.y;
  const int64_t first = (int64_t)blockIdx.x * blockDim.x;
  const int64_t last_visible = p0 + t;
  int64_t i = first + threadIdx.x;
  if (first > last_visible) {  // whole block masked
    if (i < n_entries) scores[(int64_t)t * n_entries + i] = -INFINITY;
    return;
  }
  load_qhat(q_data + (int64_t)t * kIdxHeads * kIkBytes, q_e8m0 + (int64_t)t * kIdxHeads * kIkScales, qs);
  if (threadIdx.x < kIdxHeads) ws[threadIdx.x] = w[t * kIdxHeads + threadIdx.x];
  __syncthreads();
  if (i >= n_entries) return;
  float out = -INFINITY;
  if (i <= last_visible) out = score_row(ik_data + i * kIkBytes, ik_scale + i * kIkScales, qs, ws);
  scores[(int64_t)t * n_entries + i] = out;
}

}  // namespace csa2

using namespace csa2;

int csa2_read_and_clear_index_error(cudaStream_t s) {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_index_error, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return CSA2_ERR_CUDA;
  if (cudaMemcpyToSymbolAsync(g_index_error, &z, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return CSA2_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return CSA2_ERR_CUDA;
  return v;
}

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

static int device_sm_count() {
  static int sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!sms[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    sms[dev] = v > 0 ? v : 148;
  }
  return sms[dev];
}

// Tensor-core scan of list entries 0..n_pos-1 of every sequence: cache
// positions 0..n_pos-1 (TMA tiles) or, with a positions list, the listed ones
// (gathered row by row).
int csa2_launch_index_score_tc(const uint8_t* q_data, const uint8_t* q_e8m0, const float* w, int32_t B,
                               const uint8_t* ik_data, const uint8_t* ik_scale, int64_t cap,
                               const int32_t* n_visible, const int32_t* positions, int64_t n_pos, float* scores,
                               uint32_t* hist, cudaStream_t stream) {
  if (n_pos == 0 || B == 0) return CSA2_OK;
  if (!csa2_aligned(q_data, 16) || !csa2_aligned(q_e8m0, 4)) return CSA2_ERR_ALIGNMENT;
  auto encode = tensor_map_encoder();
  if (!encode) return CSA2_ERR_CUDA;
  CUtensorMap map;
  cuuint64_t dims[3] = {(cuuint64_t)kIkBytes, (cuuint64_t)cap, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)kIkBytes, (cuuint64_t)cap * kIkBytes};
  cuuint32_t box[3] = {(cuuint32_t)kIkBytes, (cuuint32_t)scan_tc::kTileRows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, (void*)ik_data, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return CSA2_ERR_CUDA;
  // one wave of 3 CTAs per SM, each on a contiguous run of tiles of one sequence
  const int64_t tiles = (n_pos + scan_tc::kTileRows - 1) / scan_tc::kTileRows;
  const int64_t target = 3LL * device_sm_count();
  int64_t chunks = target / B;
  if (chunks < 1) chunks = 1;
  if (chunks > tiles) chunks = tiles;
  const int64_t per = (tiles + chunks - 1) / chunks;
  chunks = (tiles + per - 1) / per;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(scan_tc::index_score_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             scan_tc::kSmemBytes) != cudaSuccess)
      return CSA2_ERR_CUDA;
    attr = true;
  }
  scan_tc::Params prm{ik_data, positions, q_data, q_e8m0, w, ik_scale, cap, n_visible, n_pos, scores, (int32_t)per,
                      hist};
  scan_tc::index_score_tc_kernel<<<dim3((unsigned)chunks, (unsigned)B), scan_tc::kThreads, scan_tc::kSmemBytes,
                                   stream>>>(map, prm);
  CSA2_CHECK_LAUNCH();
  return CSA2_OK;
}

extern "C" int csa2_prefill_index_score(const uint8_t* q_data, const uint8_t* q_e8m0, const float* w,
                                        int32_t T, const uint8_t* ik_data, const uint8_t* ik_scale,
                                        int64_t n_entries, int64_t p0, float* scores, csa2_stream_t stream) {
  if (!q_data || !q_e8m0 || !w || !ik_data || !ik_scale || !scores) return CSA2_ERR_INVALID_ARG;
  if (T < 0 || n_entries < 0 || p0 < 0 || p0 + T > n_entries) return CSA2_ERR_INVALID_ARG;
  if (!csa2_aligned(ik_data, 16) || !csa2_aligned(ik_scale, 4)) return CSA2_ERR_ALIGNMENT;
  if (T == 0 || n_entries == 0) return CSA2_OK;
  dim3 grid((unsigned)((n_entries + 127) / 128), (unsigned)T);
  prefill_score_simple_kernel<<<grid, 128, 0, (cudaStream_t)stream>>>(q_data, q_e8m0, w, ik_data, ik_scale,
                                                                       n_entries, p0, scores);
  CSA2_CHECK_LAUNCH();
  return CSA2_OK;
}
