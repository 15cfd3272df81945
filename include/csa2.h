/*
 * csa2.h -- C ABI of the CSA2 sparse-attention hot path over an FP4 global
 * KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The operation follows the CSA2 layer of "DeepSeek-V4.1-Flash: Pushing the
 * Limits of KV Cache Compression" (technical report, sections 2.3, 2.3.1,
 * 2.3.2 and 2.4.4), with the sizes given in the mer.dev notes on the same
 * report (section 1 setup, section 2 byte layout, section 4):
 *   - lightning-indexer score of every visible entry,
 *       s[j] = sum_h w[h] * ReLU(q_h . k_j)   (32 heads x 128, MXFP4 q and k)
 *   - optional hierarchical candidate pool (top 2,048 blocks of 8 positions
 *     by block-max score) that restricts later Reindex layers;
 *   - Top-512 selection;
 *   - 64-head, head-dim-512 attention in which the selected 512-channel
 *     latents (E2M1 + one E4M3 scale per 16 channels) serve as both K and V,
 *     in one softmax with the 128-row FP8 sliding window of the layer.
 *
 * Conventions shared by every entry point
 *   - Every pointer is a caller-owned DEVICE pointer unless stated otherwise.
 *     No entry point allocates device memory. Scratch space is sized by the
 *     matching *_workspace_size function and passed in by the caller.
 *   - Every call is asynchronous and ordered on `stream` (a cudaStream_t;
 *     NULL is the legacy default stream). A return of CSA2_OK means the work
 *     was enqueued; errors found by the kernels themselves (an index out of
 *     range, a bounded wait that ran out) are recorded in a sticky device
 *     word that csa2_get_last_error() reads and clears.
 *   - Host-side argument checks return a negative status and enqueue nothing.
 *   - bf16 arrays are passed as `const void*` holding IEEE bfloat16 values.
 *   - Packed FP4: element 2i of a row is the low nibble of byte i, element
 *     2i+1 the high nibble.
 *   - Cache planes are struct-of-arrays, one plane per field, sequences
 *     `cap` entries apart:
 *         ik_data  [B][cap][64]  E2M1 indexer key       (64 B / entry)
 *         ik_scale [B][cap][4]   E8M0, one per 32       ( 4 B / entry)
 *         kv_data  [B][cap][256] E2M1 main-KV latent    (256 B / entry)
 *         kv_scale [B][cap][32]  E4M3, one per 16       ( 32 B / entry)
 *     which is 68 + 288 = 356 bytes per entry as in the notes' section 2.
 *     `cap` must be a multiple of CSA2_CAP_ALIGN and plane base pointers
 *     16-byte aligned; entries at positions >= n_visible[b] may hold any
 *     bytes and are never selected.
 *   - Rounding of the encoders: round-to-nearest-even, saturating at the
 *     largest finite value; inputs must be finite.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/** A cudaStream_t. */
typedef struct CUstream_st* csa2_stream_t;

/* status codes */
#define CSA2_OK 0
#define CSA2_ERR_INVALID_ARG (-1)      /* null pointer, negative size, bad value   */
#define CSA2_ERR_UNSUPPORTED_SHAPE (-2) /* a size outside what the kernels support  */
#define CSA2_ERR_ALIGNMENT (-3)        /* pointer or capacity not aligned          */
#define CSA2_ERR_CUDA (-4)             /* a CUDA runtime call or launch failed     */
#define CSA2_ERR_TIMEOUT (-5)          /* a bounded device-side wait ran out       */
#define CSA2_ERR_WORKSPACE (-6)        /* workspace too small or misaligned        */
#define CSA2_ERR_DEVICE (-7)           /* a kernel rejected an input (e.g. index)  */
#define CSA2_ERR_SCRATCH_LIMIT (-8)    /* problem needs more than the static scratch */

/* sizes fixed by the method (notes section 1 setup) */
#define CSA2_IDX_HEADS 32
#define CSA2_IDX_DIM 128
#define CSA2_HEADS 64
#define CSA2_HEAD_DIM 512
#define CSA2_TOPK 512
#define CSA2_SWA 128
#define CSA2_POOL_BLOCK 8
#define CSA2_POOL_BLOCKS 2048
#define CSA2_CAP_ALIGN 128
#define CSA2_MAX_TOPK 4096

/** Library version, major*10000 + minor*100 + patch. */
int csa2_version(void);

/** A static string naming a status code. */
const char* csa2_status_string(int status);

/**
 * Waits for `stream`, then reads and clears the sticky device error words of
 * all kernels. *device_status receives CSA2_OK or the first negative status a
 * kernel recorded. Returns CSA2_ERR_CUDA if the synchronisation failed.
 */
int csa2_get_last_error(csa2_stream_t stream, int* device_status);

/* ======================================================================== */
/* FP4 / FP8 codecs                                                          */
/* ======================================================================== */

/**
 * MXFP4 quantisation (report section 2.4.4: OCP-standard MXFP4 for indexer
 * queries and keys; notes section 2: one E8M0 scale per 32 elements).
 * x [rows][cols] bf16 -> data [rows][cols/2] packed E2M1, e8m0 [rows][cols/32].
 * Per 32-element block: X = floor(log2(amax)) - 2 clamped to [-127, 127]
 * (X = -127 for an all-zero block), scale byte X + 127, element
 * RNE_E2M1(x * 2^-X) saturating at +-6. cols must be a positive multiple of
 * 32. Errors: INVALID_ARG, UNSUPPORTED_SHAPE, CUDA.
 */
int csa2_quant_mxfp4(const void* x_bf16, int64_t rows, int32_t cols,
                     uint8_t* data, uint8_t* e8m0, csa2_stream_t stream);

/** Inverse of csa2_quant_mxfp4: out [rows][cols] fp32 = e2m1 * 2^(e - 127). */
int csa2_dequant_mxfp4(const uint8_t* data, const uint8_t* e8m0, int64_t rows,
                       int32_t cols, float* out, csa2_stream_t stream);

/**
 * Main-KV packing (report section 2.4.4: E2M1 with one E4M3 scale per 16
 * channels, NVFP4 without its second-level global scale).
 * x [n][512] bf16 -> kv_data [n][256], kv_scale [n][32].
 * Per 16-channel block: s = RNE_E4M3(amax / 6) with the quotient in IEEE
 * fp32; element RNE_E2M1(x / s) in fp32 saturating at +-6; s == 0 gives an
 * all-zero block. Errors: INVALID_ARG, CUDA.
 */
int csa2_pack_kv_fp4(const void* x_bf16, int64_t n, uint8_t* kv_data,
                     uint8_t* kv_scale, csa2_stream_t stream);

/** Inverse of csa2_pack_kv_fp4: out [n][512] bf16 = e2m1 * e4m3 (exact). */
int csa2_unpack_kv_fp4(const uint8_t* kv_data, const uint8_t* kv_scale,
                       int64_t n, void* out_bf16, csa2_stream_t stream);

/**
 * SWA KV in FP8 (report section 2.4.4, last paragraph: SWA KV stays FP8).
 * x [n] bf16 -> out [n] E4M3 bytes, RNE saturating at +-448, no scale.
 */
int csa2_pack_fp8_e4m3(const void* x_bf16, int64_t n, uint8_t* out,
                       csa2_stream_t stream);

/** Inverse of csa2_pack_fp8_e4m3: out [n] bf16 (exact). */
int csa2_unpack_fp8_e4m3(const uint8_t* in, int64_t n, void* out_bf16,
                         csa2_stream_t stream);

/**
 * Fused KV append (report section 2.4.4: the main-KV latent is quantised
 * after RoPE into E2M1 with one E4M3 scale per 16 channels, no global scale;
 * the indexer key into OCP MXFP4): T new entries per sequence, written at
 * positions n_visible[b] .. n_visible[b] + T - 1 of its planes.
 *   kv_bf16 [B][T][512] bf16 (the RoPE'd latents, 16-byte aligned),
 *   ik_bf16 [B][T][128] bf16 (the indexer keys, 16-byte aligned);
 *   kv planes [B][cap][256] / [B][cap][32] (kv_data 8-byte aligned),
 *   ik planes [B][cap][64] / [B][cap][4] (ik_data 16-byte aligned);
 *   n_visible [B] int32; n_visible_out [B] int32 (nullable) receives
 *   n_visible + T. It may be n_visible itself (advanced in place).
 * The bytes written equal csa2_pack_kv_fp4 and csa2_quant_mxfp4 of the same
 * rows. A sequence whose T entries do not fit below cap gets none of them and
 * keeps its count; csa2_get_last_error then reports DEVICE.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE (cap above 2^31-1), ALIGNMENT, CUDA.
 */
int csa2_kv_append(const void* kv_bf16, const void* ik_bf16, int32_t B,
                   int32_t T, uint8_t* kv_data, uint8_t* kv_scale,
                   uint8_t* ik_data, uint8_t* ik_scale, int64_t cap,
                   const int32_t* n_visible, int32_t* n_visible_out,
                   csa2_stream_t stream);

/**
 * Sequence compressor of the encoder's Full layers (the paperglide summary of
 * DeepSeek-V4, "Compressed Sparse Attention": every m tokens merge into one
 * compressed entry; the notes' section 4.1: CSA2 blocks do not overlap and
 * the merge is softmax-weighted). For entry e (tokens em .. em+m-1) and
 * channel c:  w_a = softmax_a( Z[em+a][c] + bias[a][c] ),
 *             entry[e][c] = sum_a w_a * C[em+a][c]   (fp32),
 * rounded to bf16 and packed as the main-KV latent (E2M1 + E4M3/16, the bytes
 * csa2_pack_kv_fp4 writes for that bf16 row).
 *   c_bf16, z_bf16 [n_tokens][512] bf16 (16-byte aligned), bias [m][512]
 *   fp32 (16-byte aligned); n_tokens a multiple of m. Entries 0 .. n_tokens/m - 1 of kv_data
 *   [..][256] (8-byte aligned) and kv_scale [..][32] are written (offset the
 *   plane pointers to append); out_bf16 [n_tokens/m][512] (nullable, 16-byte
 *   aligned) receives the bf16 entries.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE (n_tokens % m), ALIGNMENT, CUDA.
 */
int csa2_compress_kv(const void* c_bf16, const void* z_bf16, const float* bias,
                     int64_t n_tokens, int32_t m, uint8_t* kv_data,
                     uint8_t* kv_scale, void* out_bf16, csa2_stream_t stream);

/* ======================================================================== */
/* Lightning indexer, pool and Top-K                                         */
/* ======================================================================== */

/**
 * Indexer scores (report sections 2.3 and 2.3.2; notes section 4.1 and 4.4:
 * 32 x 128 multiply-adds per query-entry pair).
 *   s[b][i] = sum_h w[b][h] * ReLU( sum_c qhat[b][h][c] * khat[b][p][c] )
 * with p = i (positions == NULL) or p = positions[b][i] (a Reindex layer
 * scoring its candidate pool). qhat, khat are the MXFP4 values.
 *   q_data [B][32][64], q_e8m0 [B][32][4]  (from csa2_quant_mxfp4)
 *   w [B][32] fp32 head weights
 *   ik planes with capacity `cap`, n_visible [B] int32 (0 <= n_visible <= cap)
 *   positions [B][n_pos] int32 or NULL
 *   scores [B][n_pos] fp32 out; -inf where p < 0 or p >= n_visible[b].
 * Errors: INVALID_ARG, ALIGNMENT (cap or plane pointers), CUDA.
 */
int csa2_index_score(const uint8_t* q_data, const uint8_t* q_e8m0,
                     const float* w, int32_t B, const uint8_t* ik_data,
                     const uint8_t* ik_scale, int64_t cap,
                     const int32_t* n_visible, const int32_t* positions,
                     int64_t n_pos, float* scores, csa2_stream_t stream);

/**
 * The same scores as csa2_index_score with positions == NULL, with another
 * schedule. csa2_index_score gives each CTA a fixed range of a sequence's
 * 128-entry tiles. Here, after one fixed pipeline depth, the CTAs of a
 * sequence claim tiles two at a time from a counter, so CTAs with a larger
 * share of the memory bandwidth take more (csa2_index_topk schedules its scan
 * this way, with counters in its workspace).
 *   tile_counters [2 * B] int32, device, 8-byte aligned, owned by the caller:
 *   all zero before the first call; every call that completes leaves them
 *   zero again. Calls that may run at the same time need their own buffers.
 *   Other arguments as csa2_index_score (n_pos <= cap).
 * Errors: INVALID_ARG (also a NULL tile_counters), ALIGNMENT, CUDA.
 */
int csa2_index_score_claimed(const uint8_t* q_data, const uint8_t* q_e8m0,
                             const float* w, int32_t B, const uint8_t* ik_data,
                             const uint8_t* ik_scale, int64_t cap,
                             const int32_t* n_visible, int64_t n_pos,
                             float* scores, int32_t* tile_counters,
                             csa2_stream_t stream);

/**
 * Bytes of workspace csa2_topk needs for B rows of n scores and a given k.
 */
size_t csa2_topk_workspace_size(int32_t B, int64_t n, int32_t k);

/**
 * Top-K per row (report section 2.3: the indexer selects the Top-K entries
 * for each query; K = 512 in the notes' setup).
 *   scores [B][n] fp32; an element is a candidate when its score is neither
 *   NaN nor -inf, its column is < n_valid[b] (n_valid may be NULL) and its
 *   position is >= 0. position = positions[b][i] (or i when NULL).
 *   idx [B][k] int32 out: the positions of the k largest candidates, ties
 *   broken by smaller position, written in ascending position order and
 *   padded with -1 at the end when fewer than k candidates exist.
 * 1 <= k <= CSA2_MAX_TOPK. The result is deterministic.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, WORKSPACE, CUDA.
 */
int csa2_topk(const float* scores, int32_t B, int64_t n,
              const int32_t* n_valid, const int32_t* positions, int32_t k,
              int32_t* idx, void* workspace, size_t workspace_bytes,
              csa2_stream_t stream);

/**
 * Top-K that allocates nothing and takes no workspace: the same selection as
 * csa2_topk (same arguments, same result), with its scratch held in a fixed
 * device buffer of CSA2_TOPK_STATIC_SCRATCH_BYTES that lives inside this
 * library. The report has no counterpart of this entry point; it exists for
 * callers that may not allocate device memory at all -- for example a plugin
 * whose host engine owns every device allocation and hands it only input and
 * output buffers, or a serving loop that must not pay cudaMalloc's implicit
 * device synchronisation on its request path.
 *   - Every GPU that loads the library holds the buffer until the process
 *     exits.
 *   - The first call on a device looks up the buffer's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture. The address is kept for the life of the
 *     process: it is not valid after cudaDeviceReset, so a caller that resets
 *     a device must not call this entry point on it again.
 *   - All calls share the one buffer and it keeps the last call's contents;
 *     the call clears what must start at zero. Calls that overlap on the GPU
 *     (different streams, or different host threads) race on the buffer:
 *     order them on one stream.
 *   - Returns CSA2_ERR_SCRATCH_LIMIT when csa2_topk_workspace_size(B, n, k)
 *     exceeds CSA2_TOPK_STATIC_SCRATCH_BYTES (32 MiB: at k = 512, up to 61
 *     rows of 65,536 scores fit), and otherwise the errors of csa2_topk.
 */
#define CSA2_TOPK_STATIC_SCRATCH_BYTES (32u << 20)
int csa2_topk_static(const float* scores, int32_t B, int64_t n,
                     const int32_t* n_valid, const int32_t* positions,
                     int32_t k, int32_t* idx, csa2_stream_t stream);

/** Bytes of workspace csa2_block_pool needs. */
size_t csa2_block_pool_workspace_size(int32_t B, int64_t n, int32_t block,
                                      int32_t n_blocks);

/**
 * Hierarchical candidate pool (report section 2.3.2 and Figure 5: each block
 * takes the maximum index score among its positions; the best blocks form
 * the pool, e.g. 2,048 blocks of 8 = 16,384 positions).
 *   scores [B][n] fp32 from the Full layer's scan; block b covers positions
 *   [block*b, block*b + block) within [0, n_visible[b]).
 *   pool [B][n_blocks * block] int32 out: the positions of the n_blocks
 *   blocks with the largest block maxima (ties: smaller block id), blocks in
 *   ascending order, -1 past n_visible and in unused slots.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, WORKSPACE, CUDA.
 */
int csa2_block_pool(const float* scores, int32_t B, int64_t n,
                    const int32_t* n_visible, int32_t block, int32_t n_blocks,
                    int32_t* pool, void* workspace, size_t workspace_bytes,
                    csa2_stream_t stream);

/**
 * Block maxima (report section 2.3.2: a block's score is the maximum index
 * score among its positions).
 *   bmax[b][j] = max of the non-NaN scores[b][block*j .. block*j+block) within
 *   [0, n_visible[b]) (n_visible may be NULL: all n), -inf for none.
 *   bmax [B][ceil(n / block)] fp32 out. Errors: INVALID_ARG, CUDA.
 */
int csa2_block_max(const float* scores, int32_t B, int64_t n,
                   const int32_t* n_visible, int32_t block, float* bmax,
                   csa2_stream_t stream);

/* ======================================================================== */
/* Context sharding: the exchange steps of a step split across ranks          */
/* ======================================================================== */
/* A rank owns the contiguous entries [lo, hi) of every sequence (its planes
 * hold them at local positions 0 .. hi-lo-1). Exact because a global Top-K
 * winner is in its own range's local Top-K (report section 2.3: Top-K over
 * all entries; section 2.3.2: the best blocks likewise), and attention over
 * disjoint row sets merges by log-sum-exp (section 2.3: one softmax over the
 * selected and SWA rows). A candidate is an 8-byte pair {fp32 score, int32
 * global position}; -1 marks an empty slot (its score is -inf). */

/**
 * Candidates of a local Top-K: cand[b][j] = {scores[b][c], pos(c) + offset}
 * for c = idx[b][j], pos(c) = positions[b][c] (positions non-NULL) or c;
 * {-inf, -1} where c < 0, c >= n or pos(c) < 0.
 *   scores [B][n] fp32, positions [B][n] int32 or NULL, idx [B][k] int32
 *   columns (from csa2_topk without positions), cand [B][k] pairs out
 *   (8-byte aligned). Errors: INVALID_ARG, UNSUPPORTED_SHAPE (a position
 *   above 2^31-1), ALIGNMENT, CUDA.
 */
int csa2_topk_candidates(const float* scores, int32_t B, int64_t n,
                         const int32_t* positions, const int32_t* idx,
                         int32_t k, int64_t offset, void* cand,
                         csa2_stream_t stream);

/** Bytes of workspace csa2_topk_merge needs. */
size_t csa2_topk_merge_workspace_size(int32_t R, int32_t B, int32_t k,
                                      int32_t k_out);

/**
 * Merge of R ranks' candidates: idx[b] = the global positions of the k_out
 * best candidates of row b over all ranks, as csa2_topk orders and pads them
 * (ascending position, -1 at the end).
 *   cand [R][B][k] pairs (each rank's csa2_topk_candidates, gathered in rank
 *   order), idx [B][k_out] int32 out, 1 <= k_out <= CSA2_MAX_TOPK.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, ALIGNMENT, WORKSPACE, CUDA.
 */
int csa2_topk_merge(const void* cand, int32_t R, int32_t B, int32_t k,
                    int32_t k_out, int32_t* idx, void* workspace,
                    size_t workspace_bytes, csa2_stream_t stream);

/**
 * local_idx[b][j] = idx[b][j] - lo when lo <= idx[b][j] < hi, else -1: the
 * merged global positions that fall into this rank's range, as local ones
 * (the attention's idx).
 *   idx, local_idx [B][k] int32. Errors: INVALID_ARG, CUDA.
 */
int csa2_shard_positions(const int32_t* idx, int32_t B, int32_t k,
                         int64_t lo, int64_t hi, int32_t* local_idx,
                         csa2_stream_t stream);

/**
 * The merged pool restricted to this rank: for the global block ids
 * blocks[b][j] (-1 = unused), pool[b][j*block + r] = p - lo for the position
 * p = blocks[b][j]*block + r when lo <= p < hi and p - lo < n_visible[b]
 * (n_visible local, may be NULL), else -1.
 *   blocks [B][n_blocks] int32, pool [B][n_blocks*block] int32 out.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, CUDA.
 */
int csa2_shard_pool(const int32_t* blocks, int32_t B, int32_t n_blocks,
                    int32_t block, int64_t lo, int64_t hi,
                    const int32_t* n_visible, int32_t* pool,
                    csa2_stream_t stream);

/**
 * Merges R partial attention outputs of disjoint row sets in rank order
 * 0..R-1: out = sum_r exp(lse_r - L) / S * o_r with L = max_r lse_r,
 * S = sum_r exp(lse_r - L); lse_out = L + log S. A set with lse = -inf (no
 * rows) contributes nothing; a query-head with no rows at all gets 0, -inf.
 *   parts [R][n_q][64][512] fp32 (each rank's out_f32, 16-byte aligned),
 *   lses [R][n_q][64] fp32 (each rank's lse), out_bf16 [n_q][64][512] out
 *   (8-byte aligned), out_f32 (nullable, 16-byte aligned) and lse_out
 *   [n_q][64] (nullable). Errors: INVALID_ARG, ALIGNMENT, CUDA.
 */
int csa2_attn_merge(const float* parts, const float* lses, int32_t R,
                    int32_t n_q, void* out_bf16, float* out_f32,
                    float* lse_out, csa2_stream_t stream);

/** Bytes of workspace csa2_index_topk needs (pool_blocks 0 = no pool). */
size_t csa2_index_topk_workspace_size(int32_t B, int64_t n_pos, int32_t k,
                                      int32_t pool_blocks);

/**
 * Fused indexer scan + Top-K (+ pool): the Full-layer and Reindex-layer
 * index path of report section 2.3.1 in one call. Arguments as in
 * csa2_index_score and csa2_topk; if pool != NULL and pool_blocks > 0 the
 * call also builds the block pool [B][pool_blocks * CSA2_POOL_BLOCK] from the
 * same scores (only meaningful when positions == NULL).
 * Errors: as csa2_index_score and csa2_topk.
 */
int csa2_index_topk(const uint8_t* q_data, const uint8_t* q_e8m0,
                    const float* w, int32_t B, const uint8_t* ik_data,
                    const uint8_t* ik_scale, int64_t cap,
                    const int32_t* n_visible, const int32_t* positions,
                    int64_t n_pos, int32_t k, int32_t* idx,
                    int32_t pool_blocks, int32_t* pool, void* workspace,
                    size_t workspace_bytes, csa2_stream_t stream);

/**
 * csa2_index_topk with the indexer q given in bf16: the scan quantises it to
 * MXFP4 in its prologue with the same block encoder as csa2_quant_mxfp4 (same
 * bytes, so the same scores and indices), saving that kernel and its launch.
 *   q_bf16 [B][32][128] bf16 (16-byte aligned); the rest as csa2_index_topk.
 */
int csa2_index_topk_bf16(const void* q_bf16, const float* w, int32_t B,
                         const uint8_t* ik_data, const uint8_t* ik_scale,
                         int64_t cap, const int32_t* n_visible,
                         const int32_t* positions, int64_t n_pos, int32_t k,
                         int32_t* idx, int32_t pool_blocks, int32_t* pool,
                         void* workspace, size_t workspace_bytes,
                         csa2_stream_t stream);

/**
 * Prefill indexer scores with causal masking (report section 2.3; the
 * encoder-side prefill indexer cost in notes section 4.4 item 4).
 * T queries at positions p0 .. p0+T-1 of one sequence; query t sees entries
 * 0 .. p0+t (itself included).
 *   q_data [T][32][64] (16-byte aligned), q_e8m0 [T][32][4], w [T][32]
 *   ik planes of the sequence with n_entries >= p0 + T entries (ik_data
 *     16-byte aligned, ik_scale 4-byte aligned; no padding rows needed)
 *   scores [T][n_entries] fp32 out, -inf beyond each query's prefix.
 * Runs on the tensor cores: blocks of 32 queries against 128-entry key
 * tiles (block-scaled MXF4 products), a fp32 ReLU-weighted epilogue.
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED_SHAPE (T*32 or n_entries above
 * 2^31-1), CUDA; a bounded device wait that runs out is reported by
 * csa2_get_last_error as TIMEOUT.
 */
int csa2_prefill_index_score(const uint8_t* q_data, const uint8_t* q_e8m0,
                             const float* w, int32_t T,
                             const uint8_t* ik_data, const uint8_t* ik_scale,
                             int64_t n_entries, int64_t p0, float* scores,
                             csa2_stream_t stream);

/**
 * Prefill indexer scores over compressed entries (notes section 4.4 item 4:
 * the encoder's Full layers score each query against the visible compressed
 * entries, about 3,072 N^2 multiply-adds at m = 2): as
 * csa2_prefill_index_score with p0 the token position of query 0 and m tokens
 * per entry; query t sees the complete entries j < floor((p0 + t + 1) / m).
 * m = 1 is csa2_prefill_index_score. Requires floor((p0 + T) / m) <= n_entries.
 * Errors: as csa2_prefill_index_score.
 */
int csa2_prefill_index_score_compressed(const uint8_t* q_data,
                                        const uint8_t* q_e8m0, const float* w,
                                        int32_t T, const uint8_t* ik_data,
                                        const uint8_t* ik_scale,
                                        int64_t n_entries, int64_t p0,
                                        int32_t m, float* scores,
                                        csa2_stream_t stream);

/* ======================================================================== */
/* Sparse attention                                                          */
/* ======================================================================== */

/** Bytes of workspace the attention entry points need for n_queries
 *  (query-layers in decode, queries in prefill). */
size_t csa2_sparse_attn_workspace_size(int32_t n_queries, int32_t k,
                                       int32_t n_swa);

/** Kernel launches one attention call makes for n_queries on the current
 *  device (one per batch of up to 256 queries); 0 for invalid sizes. */
int csa2_sparse_attn_kernel_launches(int32_t n_queries, int32_t k,
                                     int32_t n_swa);

/**
 * Sparse decode attention (report section 2.3: each query attends to the
 * selected entries together with the layer-local SWA KV; section 2.3.1:
 * Reuse layers use the Top-K of the preceding indexing layer with their own
 * query and SWA KV; notes section 1: 64 heads of dim 512, the 512-dim latent
 * shared as K and V).
 *   q [B][L][64][512] bf16: the L layers of sequence b share idx[b]
 *     (L = 1 for one layer, 4 for 1 Full + 3 Reuse).
 *   kv planes with capacity cap; n_visible [B]; idx [B][k] int32 positions
 *     (-1 entries are skipped; a position >= n_visible[b] is a device error).
 *   swa [B][L][n_swa][512] E4M3 bytes (0 <= n_swa <= 512).
 *   S = sm_scale * q . row over the k selected rows and the n_swa SWA rows,
 *   one softmax, out = P . rows.
 *   out [B][L][64][512] bf16; out_f32 (nullable) the same before the bf16
 *   rounding; lse (nullable) [B][L][64] natural-log sum of exp(S), -inf for
 *   a query with no rows (its output is 0).
 *   k <= CSA2_MAX_TOPK, n_swa <= 512. q, swa and out_f32 16-byte aligned,
 *   out 8-byte aligned, the planes 16-byte aligned as in the conventions above.
 *   q and the swa rows are read before this call waits for the kernel just
 *   before it on the stream (the indices and n_visible are read after): they
 *   must not be written by that kernel when it is one of this library's
 *   attention or merge kernels (which let their successor start early); the
 *   packers and anything launched without programmatic dependence are safe.
 *   Precision: rows and q enter the tensor cores as fp16 (exact: the row
 *   values have at most 6 significant bits, q is scaled by a power of two per
 *   head), P as fp16 (relative rounding 2^-11), fp32 accumulation.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, ALIGNMENT, WORKSPACE, CUDA.
 */
int csa2_sparse_attn_decode(const void* q_bf16, int32_t B, int32_t L,
                            const uint8_t* kv_data, const uint8_t* kv_scale,
                            int64_t cap, const int32_t* n_visible,
                            const int32_t* idx, int32_t k, const uint8_t* swa,
                            int32_t n_swa, float sm_scale, void* out_bf16,
                            float* out_f32, float* lse, void* workspace,
                            size_t workspace_bytes, csa2_stream_t stream);

/**
 * Fused Reuse-layer decode attention (report section 2.3.1: the Reuse layers
 * of a sequence attend to the selection of its Full layer, each with its own
 * query and SWA KV; notes section 4.2: they share that selection): the same
 * arguments, results and limits as csa2_sparse_attn_decode, computed with one
 * cluster of CTAs per sequence in which every 128-row tile of selected
 * entries is gathered and dequantised once per pair of layers (once for all
 * L when L is odd) instead of once per layer. The partials of one layer are
 * the same as csa2_sparse_attn_decode's and are merged in the same order, so
 * the outputs are bit-identical to that call's.
 * When to use it: the per-layer call spreads the layers over more CTAs and
 * is faster at small batches; this call does less gather and dequantisation
 * work and is faster once the per-layer call fills the device several times
 * over (measured on GB300 at k = 512, 128 SWA rows: L = 2, B = 64: 81 vs
 * 91 us; L = 4 only at parity from B = 64).
 * Errors: those of csa2_sparse_attn_decode, and UNSUPPORTED_SHAPE when one
 * cluster (at most 8 CTAs) cannot hold the merge of the L x 64 (layer, head)
 * rows: L > 8, or k and n_swa so large that the tiles' (max, sum) pairs do
 * not fit its table ((ceil(k/128) + ceil(n_swa/128)) * ceil(64 L / C) > 576
 * for the cluster size C = min(8, the sequence's work items)).
 */
int csa2_sparse_attn_reuse(const void* q_bf16, int32_t B, int32_t L,
                           const uint8_t* kv_data, const uint8_t* kv_scale,
                           int64_t cap, const int32_t* n_visible,
                           const int32_t* idx, int32_t k, const uint8_t* swa,
                           int32_t n_swa, float sm_scale, void* out_bf16,
                           float* out_f32, float* lse, void* workspace,
                           size_t workspace_bytes, csa2_stream_t stream);

/**
 * Sparse prefill attention: T queries of one sequence, each with its own
 * Top-K and its own causal SWA window.
 *   q [T][64][512] bf16; kv planes of the sequence with n_entries entries;
 *   idx [T][k]; swa [T + n_swa - 1][512] E4M3 where query t uses rows
 *   t .. t + n_swa - 1 (the last one is the query's own position).
 *   out/out_f32/lse as in csa2_sparse_attn_decode with [T] leading.
 * Errors: as csa2_sparse_attn_decode.
 */
int csa2_sparse_attn_prefill(const void* q_bf16, int32_t T,
                             const uint8_t* kv_data, const uint8_t* kv_scale,
                             int64_t n_entries, const int32_t* idx, int32_t k,
                             const uint8_t* swa, int32_t n_swa, float sm_scale,
                             void* out_bf16, float* out_f32, float* lse,
                             void* workspace, size_t workspace_bytes,
                             csa2_stream_t stream);

/**
 * Sparse prefill attention with the Bounded-Replay SWA mask (notes section 6:
 * after the SWA cache of a prefix was evicted, only the last n_win tokens are
 * replayed and the sliding window is cut at the replay start s, so the query
 * at position i sees SWA positions [max(s, i - W + 1), i]).
 *   As csa2_sparse_attn_prefill, with replay_row >= 0 the first row of the swa
 *   array inside the replay segment: query t uses rows
 *   max(t, replay_row) .. t + n_swa - 1. With swa row r holding position
 *   p0 - (n_swa - 1) + r, replay_row = s - p0 + n_swa - 1 (0: no truncation).
 * Errors: as csa2_sparse_attn_decode.
 */
int csa2_sparse_attn_prefill_replay(const void* q_bf16, int32_t T,
                                    const uint8_t* kv_data,
                                    const uint8_t* kv_scale, int64_t n_entries,
                                    const int32_t* idx, int32_t k,
                                    const uint8_t* swa, int32_t n_swa,
                                    int32_t replay_row, float sm_scale,
                                    void* out_bf16, float* out_f32, float* lse,
                                    void* workspace, size_t workspace_bytes,
                                    csa2_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
