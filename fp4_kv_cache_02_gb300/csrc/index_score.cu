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
// Both scans run on the tensor cores: the decode scan over contiguous entries
// or a positions list of a Reindex layer (index_score_tc.cuh), and the causal
// prefill scan of a chunk of queries (prefill_score_tc.cuh).
#include "common.cuh"

namespace csa2 {

__device__ int g_index_error = 0;

}  // namespace csa2

#include "index_score_tc.cuh"
#include "prefill_score_tc.cuh"

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
// (gathered row by row). early_reads: the kernel just before in the stream
// writes nothing the scan reads (it only clears the Top-K workspace), so the
// scan's loads may start before that kernel ends.
int csa2_launch_index_score_tc(const uint8_t* q_data, const uint8_t* q_e8m0, const float* w, int32_t B,
                               const uint8_t* ik_data, const uint8_t* ik_scale, int64_t cap,
                               const int32_t* n_visible, const int32_t* positions, int64_t n_pos, float* scores,
                               uint32_t* hist, float* bmax, int early_reads, const void* q_bf16,
                               int32_t* tile_ctr, int32_t tile_ctr_stride, int32_t* tile_done,
                               cudaStream_t stream) {
  if (n_pos == 0 || B == 0) return CSA2_OK;
  if (q_bf16 ? !csa2_aligned(q_bf16, 16) : (!csa2_aligned(q_data, 16) || !csa2_aligned(q_e8m0, 4)))
    return CSA2_ERR_ALIGNMENT;
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
  static Csa2PerDeviceOnce optin;
  if (csa2_smem_optin((const void*)scan_tc::index_score_tc_kernel, scan_tc::kSmemBytes, optin) != CSA2_OK)
    return CSA2_ERR_CUDA;
  // claimed tiles (dense mode with counters): a fixed first range of one
  // pipeline's depth, then claims of two tiles
  scan_tc::Params prm{ik_data, positions, q_data, q_e8m0, w, ik_scale, cap, n_visible, n_pos, scores, (int32_t)per,
                      hist, positions ? nullptr : bmax, early_reads, (const uint16_t*)q_bf16,
                      positions ? nullptr : tile_ctr, tile_ctr_stride, scan_tc::kStages, 2,
                      positions ? nullptr : tile_done};
  CSA2_LAUNCH_PDL(scan_tc::index_score_tc_kernel, dim3((unsigned)B, (unsigned)chunks), dim3(scan_tc::kThreads),
                  (size_t)scan_tc::kSmemBytes, stream, map, prm);
  return CSA2_OK;
}

extern "C" int csa2_prefill_index_score_compressed(const uint8_t* q_data, const uint8_t* q_e8m0, const float* w,
                                                   int32_t T, const uint8_t* ik_data, const uint8_t* ik_scale,
                                                   int64_t n_entries, int64_t p0, int32_t m, float* scores,
                                                   csa2_stream_t stream) {
  if (!q_data || !q_e8m0 || !w || !ik_data || !ik_scale || !scores) return CSA2_ERR_INVALID_ARG;
  if (T < 0 || n_entries < 0 || p0 < 0 || m < 1 || (p0 + T) / m > n_entries) return CSA2_ERR_INVALID_ARG;
  if (!csa2_aligned(ik_data, 16) || !csa2_aligned(ik_scale, 4) || !csa2_aligned(q_data, 16) ||
      !csa2_aligned(q_e8m0, 4) || !csa2_aligned(w, 4))
    return CSA2_ERR_ALIGNMENT;
  if ((int64_t)T * kIdxHeads > 0x7FFFFFFFLL || n_entries > 0x7FFFFFFFLL) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (T == 0 || n_entries == 0) return CSA2_OK;
  auto encode = tensor_map_encoder();
  if (!encode) return CSA2_ERR_CUDA;
  using namespace prefill_tc;
  CUtensorMap map_ik, map_q;
  cuuint64_t kdims[2] = {(cuuint64_t)kIkBytes, (cuuint64_t)n_entries};
  cuuint64_t kstr[1] = {(cuuint64_t)kIkBytes};
  cuuint32_t kbox[2] = {(cuuint32_t)kIkBytes, (cuuint32_t)kTileRows};
  cuuint64_t qdims[2] = {(cuuint64_t)kIkBytes, (cuuint64_t)T * kIdxHeads};
  cuuint32_t qbox[2] = {(cuuint32_t)kIkBytes, 256};
  cuuint32_t estr[2] = {1, 1};
  if (encode(&map_ik, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, (void*)ik_data, kdims, kstr, kbox, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      encode(&map_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, (void*)q_data, qdims, kstr, qbox, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return CSA2_ERR_CUDA;
  static Csa2PerDeviceOnce optin;
  if (csa2_smem_optin((const void*)prefill_score_tc_kernel, kSmemBytes, optin) != CSA2_OK) return CSA2_ERR_CUDA;
  const int64_t tiles = (n_entries + kTileRows - 1) / kTileRows;
  dim3 grid((unsigned)((tiles + kChunkTiles - 1) / kChunkTiles), (unsigned)((T + kQBlock - 1) / kQBlock));
  Params prm{q_e8m0, w, ik_scale, n_entries, p0, T, m, scores};
  prefill_score_tc_kernel<<<grid, kThreads, kSmemBytes, (cudaStream_t)stream>>>(map_ik, map_q, prm);
  CSA2_CHECK_LAUNCH();
  return CSA2_OK;
}

extern "C" int csa2_prefill_index_score(const uint8_t* q_data, const uint8_t* q_e8m0, const float* w,
                                        int32_t T, const uint8_t* ik_data, const uint8_t* ik_scale,
                                        int64_t n_entries, int64_t p0, float* scores, csa2_stream_t stream) {
  return csa2_prefill_index_score_compressed(q_data, q_e8m0, w, T, ik_data, ik_scale, n_entries, p0, 1, scores,
                                             stream);
}
