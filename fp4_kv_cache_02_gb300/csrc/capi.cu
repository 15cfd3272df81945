// capi.cu -- C entry points that compose the kernels: argument checks,
// workspace carving and the fused indexer -> Top-K (-> pool) path.
#include "common.cuh"

// launchers defined in the kernel units
int csa2_launch_index_score_tc(const uint8_t* q_data, const uint8_t* q_e8m0, const float* w, int32_t B,
                               const uint8_t* ik_data, const uint8_t* ik_scale, int64_t cap,
                               const int32_t* n_visible, const int32_t* positions, int64_t n_pos, float* scores,
                               uint32_t* hist, float* bmax, int early_reads, const void* q_bf16,
                               int32_t* tile_ctr, int32_t tile_ctr_stride, int32_t* tile_done,
                               cudaStream_t stream);
int csa2_topk_prepare(int32_t B, int64_t n, int32_t k, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream, uint32_t** hist, int32_t** scan_ctr, int32_t* scan_ctr_stride);
int csa2_topk_from_hist(const float* scores, int32_t B, int64_t n, const int32_t* n_valid, const int32_t* positions,
                        int32_t k, int32_t* idx, void* workspace, cudaStream_t stream);
int csa2_launch_topk(const float* scores, int32_t B, int64_t n, const int32_t* n_valid, const int32_t* positions,
                     int32_t k, int32_t* idx, void* workspace, size_t workspace_bytes, cudaStream_t stream);
int csa2_launch_block_pool(const float* scores, int32_t B, int64_t n, const int32_t* n_visible, int32_t block,
                           int32_t n_blocks, int32_t* pool, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);
int csa2_launch_pool_from_bmax(const float* bmax, int32_t B, int64_t n, const int32_t* n_visible, int32_t block,
                               int32_t n_blocks, int32_t* pool, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);

extern "C" int csa2_version(void) { return 100; }

extern "C" const char* csa2_status_string(int status) {
  switch (status) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARG: return "invalid argument";
    case CSA2_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case CSA2_ERR_ALIGNMENT: return "misaligned pointer or capacity";
    case CSA2_ERR_CUDA: return "CUDA runtime error";
    case CSA2_ERR_TIMEOUT: return "bounded device wait ran out";
    case CSA2_ERR_WORKSPACE: return "workspace too small or misaligned";
    case CSA2_ERR_DEVICE: return "a kernel rejected an input";
    case CSA2_ERR_SCRATCH_LIMIT: return "problem needs more than the static scratch buffer";
    default: return "unknown status";
  }
}

extern "C" int csa2_get_last_error(csa2_stream_t stream, int* device_status) {
  if (!device_status) return CSA2_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaStreamSynchronize(s) != cudaSuccess) return CSA2_ERR_CUDA;
  int first = CSA2_OK;
  int (*readers[])(cudaStream_t) = {csa2_read_and_clear_codec_error, csa2_read_and_clear_index_error,
                                    csa2_read_and_clear_topk_error, csa2_read_and_clear_attn_error};
  for (auto rd : readers) {
    int v = rd(s);
    if (v == CSA2_ERR_CUDA) return CSA2_ERR_CUDA;
    if (first == CSA2_OK && v != CSA2_OK) first = v;
  }
  *device_status = first;
  return CSA2_OK;
}

static int check_index_args(const uint8_t* q_data, const uint8_t* q_e8m0, const float* w, int32_t B,
                            const uint8_t* ik_data, const uint8_t* ik_scale, int64_t cap, const int32_t* n_visible,
                            int64_t n_pos) {
  if (!q_data || !q_e8m0 || !w || !ik_data || !ik_scale || !n_visible) return CSA2_ERR_INVALID_ARG;
  if (B < 0 || cap < 0 || n_pos < 0) return CSA2_ERR_INVALID_ARG;
  if (cap % CSA2_CAP_ALIGN) return CSA2_ERR_ALIGNMENT;
  if (!csa2_aligned(ik_data, 16) || !csa2_aligned(ik_scale, 16)) return CSA2_ERR_ALIGNMENT;
  if (n_pos > 0x7FFFFFFFLL || cap > 0x7FFFFFFFLL) return CSA2_ERR_UNSUPPORTED_SHAPE;
  return CSA2_OK;
}

extern "C" int csa2_index_score(const uint8_t* q_data, const uint8_t* q_e8m0, const float* w, int32_t B,
                                const uint8_t* ik_data, const uint8_t* ik_scale, int64_t cap,
                                const int32_t* n_visible, const int32_t* positions, int64_t n_pos, float* scores,
                                csa2_stream_t stream) {
  int rc = check_index_args(q_data, q_e8m0, w, B, ik_data, ik_scale, cap, n_visible, n_pos);
  if (rc) return rc;
  if (!scores) return CSA2_ERR_INVALID_ARG;
  if (positions == nullptr && n_pos > cap) return CSA2_ERR_INVALID_ARG;
  if (positions && !csa2_aligned(positions, 4)) return CSA2_ERR_ALIGNMENT;
  return csa2_launch_index_score_tc(q_data, q_e8m0, w, B, ik_data, ik_scale, cap, n_visible, positions, n_pos, scores,
                                    nullptr, nullptr, 0, nullptr, nullptr, 0, nullptr, (cudaStream_t)stream);
}

extern "C" int csa2_index_score_claimed(const uint8_t* q_data, const uint8_t* q_e8m0, const float* w, int32_t B,
                                        const uint8_t* ik_data, const uint8_t* ik_scale, int64_t cap,
                                        const int32_t* n_visible, int64_t n_pos, float* scores,
                                        int32_t* tile_counters, csa2_stream_t stream) {
  int rc = check_index_args(q_data, q_e8m0, w, B, ik_data, ik_scale, cap, n_visible, n_pos);
  if (rc) return rc;
  if (!scores || !tile_counters || n_pos > cap) return CSA2_ERR_INVALID_ARG;
  if (!csa2_aligned(tile_counters, 8)) return CSA2_ERR_ALIGNMENT;
  // sequence b's counter and finished-CTA count: tile_counters[2b], [2b + 1]
  return csa2_launch_index_score_tc(q_data, q_e8m0, w, B, ik_data, ik_scale, cap, n_visible, nullptr, n_pos, scores,
                                    nullptr, nullptr, 0, nullptr, tile_counters, 2, tile_counters + 1,
                                    (cudaStream_t)stream);
}

static inline size_t al256(size_t x) { return (x + 255) / 256 * 256; }

extern "C" size_t csa2_index_topk_workspace_size(int32_t B, int64_t n_pos, int32_t k, int32_t pool_blocks) {
  if (B <= 0 || n_pos < 0 || k <= 0) return 0;
  size_t scores = al256((size_t)B * (size_t)(n_pos > 0 ? n_pos : 1) * 4);
  size_t t = csa2_topk_workspace_size(B, n_pos, k);
  if (pool_blocks > 0) {
    // block maxima (written by the scan) get their own slice; the pool's
    // Top-K reuses the Full Top-K's scratch after it
    scores += al256((size_t)B * (size_t)((n_pos + CSA2_POOL_BLOCK - 1) / CSA2_POOL_BLOCK + 1) * 4);
    size_t p = csa2_block_pool_workspace_size(B, n_pos, CSA2_POOL_BLOCK, pool_blocks);
    if (p > t) t = p;
  }
  return scores + t;
}

static int index_topk(const uint8_t* q_data, const uint8_t* q_e8m0, const void* q_bf16, const float* w, int32_t B,
                      const uint8_t* ik_data, const uint8_t* ik_scale, int64_t cap, const int32_t* n_visible,
                      const int32_t* positions, int64_t n_pos, int32_t k, int32_t* idx, int32_t pool_blocks,
                      int32_t* pool, void* workspace, size_t workspace_bytes, csa2_stream_t stream) {
  int rc = q_bf16 ? check_index_args((const uint8_t*)q_bf16, (const uint8_t*)q_bf16, w, B, ik_data, ik_scale, cap,
                                     n_visible, n_pos)
                  : check_index_args(q_data, q_e8m0, w, B, ik_data, ik_scale, cap, n_visible, n_pos);
  if (rc) return rc;
  if (!idx) return CSA2_ERR_INVALID_ARG;
  if (k <= 0 || k > CSA2_MAX_TOPK || pool_blocks < 0 || pool_blocks > CSA2_MAX_TOPK)
    return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (positions == nullptr && n_pos > cap) return CSA2_ERR_INVALID_ARG;
  if (pool_blocks > 0 && (!pool || positions)) return CSA2_ERR_INVALID_ARG;
  if (positions && !csa2_aligned(positions, 4)) return CSA2_ERR_ALIGNMENT;
  size_t need = csa2_index_topk_workspace_size(B, n_pos, k, pool_blocks);
  if (!workspace || workspace_bytes < need || !csa2_aligned(workspace, 256)) return CSA2_ERR_WORKSPACE;
  if (B == 0) return CSA2_OK;
  cudaStream_t s = (cudaStream_t)stream;
  float* scores = (float*)workspace;
  size_t off = al256((size_t)B * (size_t)(n_pos > 0 ? n_pos : 1) * 4);
  float* bmax = nullptr;
  if (pool_blocks > 0) {
    bmax = (float*)((char*)workspace + off);
    off += al256((size_t)B * (size_t)((n_pos + CSA2_POOL_BLOCK - 1) / CSA2_POOL_BLOCK + 1) * 4);
  }
  char* rest = (char*)workspace + off;
  size_t rest_bytes = workspace_bytes - off;
  // the scan's epilogue builds the Top-K histogram (and the pool's block maxima)
  uint32_t* hist = nullptr;
  int32_t* scan_ctr = nullptr;
  int32_t scan_ctr_stride = 0;
  rc = csa2_topk_prepare(B, n_pos, k, rest, rest_bytes, s, &hist, &scan_ctr, &scan_ctr_stride);
  if (rc) return rc;
  rc = csa2_launch_index_score_tc(q_data, q_e8m0, w, B, ik_data, ik_scale, cap, n_visible, positions, n_pos, scores,
                                  hist, bmax, 1, q_bf16, scan_ctr, scan_ctr_stride, nullptr,
                                  s);  // just after the workspace clear
  if (rc) return rc;
  rc = csa2_topk_from_hist(scores, B, n_pos, positions ? nullptr : n_visible, positions, k, idx, rest, s);
  if (rc) return rc;
  if (pool_blocks > 0)
    rc = csa2_launch_pool_from_bmax(bmax, B, n_pos, n_visible, CSA2_POOL_BLOCK, pool_blocks, pool, rest, rest_bytes, s);
  return rc;
}

extern "C" int csa2_index_topk(const uint8_t* q_data, const uint8_t* q_e8m0, const float* w, int32_t B,
                               const uint8_t* ik_data, const uint8_t* ik_scale, int64_t cap,
                               const int32_t* n_visible, const int32_t* positions, int64_t n_pos, int32_t k,
                               int32_t* idx, int32_t pool_blocks, int32_t* pool, void* workspace,
                               size_t workspace_bytes, csa2_stream_t stream) {
  return index_topk(q_data, q_e8m0, nullptr, w, B, ik_data, ik_scale, cap, n_visible, positions, n_pos, k, idx,
                    pool_blocks, pool, workspace, workspace_bytes, stream);
}

extern "C" int csa2_index_topk_bf16(const void* q_bf16, const float* w, int32_t B, const uint8_t* ik_data,
                                    const uint8_t* ik_scale, int64_t cap, const int32_t* n_visible,
                                    const int32_t* positions, int64_t n_pos, int32_t k, int32_t* idx,
                                    int32_t pool_blocks, int32_t* pool, void* workspace, size_t workspace_bytes,
                                    csa2_stream_t stream) {
  if (!q_bf16) return CSA2_ERR_INVALID_ARG;
  return index_topk(nullptr, nullptr, q_bf16, w, B, ik_data, ik_scale, cap, n_visible, positions, n_pos, k, idx,
                    pool_blocks, pool, workspace, workspace_bytes, stream);
}
