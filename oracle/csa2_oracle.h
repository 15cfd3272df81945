/*
 * csa2_oracle.h -- plain CPU oracle for the CSA2 sparse-attention hot path.
 *
 * TEST INFRASTRUCTURE. Only tests/, the smoke check in __graft_entry__.py and
 * the cpu_baseline leg of bench.py may load or call this code. The CUDA
 * library never links it and shares no code, header, table or helper with it;
 * the two sides agree only on the byte layout of the packed planes.
 *
 * Sources (cited by short tag below and in csa2_oracle.c):
 *   [R]  "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression"
 *        (technical-report digest, arXiv 2609.19969)
 *   [B]  "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression"
 *        (mer.dev reading notes on the same report)
 *   [V4] "DeepSeek-V4: Towards Highly Efficient Million-Token Context
 *        Intelligence" (paperglide summary)
 *
 * Packed layouts (element 2i in the low nibble, 2i+1 in the high nibble):
 *   indexer K / indexer q, MXFP4 ([R] 2.4.4, [B] 2): per row of 128 values,
 *     64 bytes of E2M1 codes + 4 bytes of E8M0 scales (one per 32 values) = 68 B.
 *   main KV ([R] 2.4.4, [B] 2 and 5): per 512-channel latent,
 *     256 bytes of E2M1 codes + 32 bytes of E4M3 scales (one per 16) = 288 B.
 *   SWA KV ([R] 2.4.4): one E4M3 byte per channel, no scale.
 */
#ifndef CSA2_ORACLE_H
#define CSA2_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- element formats -------------------------------------------------- */
double orc_e2m1_value(unsigned code);      /* 4-bit code -> value            */
double orc_e4m3_value(unsigned code);      /* 8-bit code -> value (NaN 0x7F) */
double orc_e8m0_value(unsigned code);      /* 8-bit code -> 2^(code-127)     */
unsigned orc_e2m1_encode(float x);         /* RNE, saturating at +-6         */
unsigned orc_e4m3_encode(float x);         /* RNE, saturating at +-448       */

/* ---- codecs over arrays ----------------------------------------------- */
void orc_quant_mxfp4(const float* x, int64_t rows, int cols,
                     uint8_t* data, uint8_t* e8m0);
void orc_dequant_mxfp4(const uint8_t* data, const uint8_t* e8m0,
                       int64_t rows, int cols, double* out);
void orc_pack_kv_fp4(const float* x, int64_t n, uint8_t* kv_data,
                     uint8_t* kv_scale);
void orc_unpack_kv_fp4(const uint8_t* kv_data, const uint8_t* kv_scale,
                       int64_t n, double* out);
void orc_pack_fp8(const float* x, int64_t n, uint8_t* out);
void orc_unpack_fp8(const uint8_t* in, int64_t n, double* out);

/* ---- byte arithmetic --------------------------------------------------- */
int orc_main_kv_entry_bytes(void);   /* 288 */
int orc_indexer_k_entry_bytes(void); /* 68  */

/* ---- lightning-indexer score --------------------------------------------
 * s[i] = sum_h w[h] * max(0, sum_c qhat[h][c] * khat[p_i][c]) for the n rows
 * p_i = positions[i] (positions == NULL means p_i = i; p_i < 0 gives s = -inf).
 * q: [32][64] codes + [32][4] scales. k planes: [*][64] + [*][4].
 * out32 receives the fp32 rounding of the double sum; out64 (nullable) the
 * double itself. Returns the number of multiply-accumulates performed.     */
uint64_t orc_index_score(const uint8_t* q_data, const uint8_t* q_e8m0,
                         const float* w, const uint8_t* ik_data,
                         const uint8_t* ik_scale, const int32_t* positions,
                         int64_t n, float* out32, double* out64);

/* ---- Top-K ----------------------------------------------------------------
 * The k largest scores, ordered by (score desc, position asc). Entries with a
 * negative position or score -inf are not candidates. idx receives positions
 * (positions[i], or i when positions == NULL), padded with -1. Returns the
 * number of valid outputs.                                                  */
int orc_topk(const float* scores, const int32_t* positions, int64_t n, int k,
             int32_t* idx);

/* ---- hierarchical block pool -----------------------------------------------
 * Block b covers positions [block*b, block*b+block) within [0, n). Its score
 * is the max over those positions. The n_blocks best blocks by
 * (max desc, b asc) are kept; pool lists their positions in ascending order,
 * -1 where a block runs past n and for unused slots. Returns blocks kept.   */
int orc_block_pool(const float* scores, int64_t n, int block, int n_blocks,
                   int32_t* pool);

/* Block maxima alone: bmax[b] = max of scores over block b within [0, n)
 * (NaN skipped), -inf for a block with no score.                           */
void orc_block_max(const float* scores, int64_t n, int block, float* bmax);

/* ---- sparse attention -----------------------------------------------------
 * One query: q [H][D] (values already bf16-exact), rows = dequantised main KV
 * of idx[0..k) (negative entries skipped) followed by the n_swa SWA rows.
 * S = sm_scale * q . row ; one softmax over all rows ; out = P . rows.
 * out [H][D] and lse [H] (natural log; -inf when there is no row).          */
void orc_sparse_attn(const float* q, int H, int D, const uint8_t* kv_data,
                     const uint8_t* kv_scale, const int32_t* idx, int k,
                     const uint8_t* swa, int n_swa, double sm_scale,
                     double* out, double* lse);

/* ---- sequence compressor (CSA: every m tokens merge into one entry; CSA2
 * blocks do not overlap; softmax-weighted merge). For entry e and channel c:
 * w_a = softmax over a = 0..m-1 of Z[em+a][c] + bias[a][c];
 * out[e][c] = sum_a w_a C[em+a][c]. C, Z [n_tokens][D], bias [m][D],
 * out [n_tokens/m][D], all in double.                                       */
void orc_compress_kv(const double* C, const double* Z, const double* bias,
                     int64_t n_tokens, int m, int D, double* out);

/* ---- merge of attention over disjoint row sets ------------------------------
 * R partial results (out_r [H][D], lse_r [H]) of one query, each the softmax
 * attention over its own rows, merged into the attention over the union of
 * the rows: since softmax weights over the union are exp(s - LSE) with
 * LSE = log sum_r exp(lse_r), out = sum_r exp(lse_r - LSE) * out_r.
 * A set with lse = -inf has no rows; all -inf gives out 0, lse -inf.        */
void orc_attn_merge(const double* outs, const double* lses, int R, int H,
                    int D, double* out, double* lse);

/* ---- whole decode step for a batch (the timed CPU baseline) --------------
 * For each of the B sequences (OpenMP over sequences): score all n_visible[b]
 * entries, Top-k, then attention for each of the L layers that share the
 * indices (layer 0 = the indexing layer, 1..L-1 = Reuse layers).
 * Layouts: q_data [B][32][64], q_e8m0 [B][32][4], w [B][32],
 * ik planes [B][cap][64|4], kv planes [B][cap][256|32], Q [B][L][H][D] floats,
 * swa [B][L][n_swa][D] bytes; outputs idx [B][k], out [B][L][H][D].
 * Returns total multiply-accumulates of the scoring stage.                  */
uint64_t orc_decode_batch(int B, int64_t cap, const int32_t* n_visible,
                          const uint8_t* q_data, const uint8_t* q_e8m0,
                          const float* w, const uint8_t* ik_data,
                          const uint8_t* ik_scale, const uint8_t* kv_data,
                          const uint8_t* kv_scale, int k, int L,
                          const float* Q, int H, int D, const uint8_t* swa,
                          int n_swa, double sm_scale, int32_t* idx,
                          double* out, int n_threads);

int orc_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif
