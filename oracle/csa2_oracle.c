/*
 * csa2_oracle.c -- plain, slow CPU oracle for the CSA2 hot path.
 *
 * TEST INFRASTRUCTURE (see csa2_oracle.h): only tests/, the smoke check and
 * bench.py's cpu_baseline leg use it. Nothing here is blocked, fused or
 * reordered beyond the definitions it cites; floating point is accumulated in
 * double and rounded once where an fp32 result is produced.
 *
 * Readings taken where the pages leave a step open (each also listed in the
 * design notes of the repository):
 *  - E2M1 / E4M3 / E8M0 are the OCP microscaling element and scale formats the
 *    pages name ([R] 2.4.4 "OCP-standard MXFP4"; "E2M1 with one E4M3 scale per
 *    16 channels, following NVFP4 ... omitting its second-level global scale").
 *  - Rounding is round-to-nearest-even with saturation; the sign of a value
 *    that rounds to zero is kept. The pages print no rounding rule and the
 *    block quantiser formula in [B] 5 was lost in extraction.
 *  - MXFP4 shared exponent: X = floor(log2(amax)) - 2 (the largest E2M1
 *    exponent), clamped to [-127, 127]; an all-zero block gets X = -127.
 *  - Main-KV scale: s = RNE_E4M3(amax / 6) with the quotient taken in IEEE
 *    fp32; elements RNE_E2M1(x / s) in fp32; s == 0 gives an all-zero block.
 *  - Indexer score s = sum_h w_h ReLU(q_h . k) over the 32 heads, with q and k
 *    both MXFP4 ([R] 2.4.4: FP4 indexer queries and keys; [B] 4.1: the
 *    multi-head ReLU-weighted sum carried over from DSA/V4), no 1/sqrt(d).
 *  - Top-K ties are broken by ascending position.
 */
#include "csa2_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_IDX_HEADS 32   /* [B] 1: indexer has 32 heads of dim 128 */
#define ORC_IDX_DIM 128
#define ORC_MX_BLOCK 32    /* [B] 2: one E8M0 scale per 32 elements */
#define ORC_KV_DIM 512     /* [B] 1: 512-dim KV latent */
#define ORC_KV_BLOCK 16    /* [R] 2.4.4: one E4M3 scale per 16 channels */

/* ------------------------------------------------------------------------ */
/* Element formats ([R] 2.4.4; OCP MX element/scale definitions)             */
/* ------------------------------------------------------------------------ */

/* E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 * Exponent 0 is subnormal: value = m * 0.5. */
double orc_e2m1_value(unsigned code) {
  unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
  double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
  return s ? -mag : mag;
}

/* E4M3 (the "FN" variant): bias 7, no infinities, S.1111.111 is NaN.
 * Exponent 0 is subnormal: value = (m/8) * 2^-6. Largest finite is 448. */
double orc_e4m3_value(unsigned code) {
  unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
  double mag;
  if (e == 15u && m == 7u) return NAN;
  mag = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, (int)e - 7);
  return s ? -mag : mag;
}

/* E8M0: a bare biased exponent, 2^(code-127); 0xFF is NaN. */
double orc_e8m0_value(unsigned code) {
  if ((code & 0xFFu) == 0xFFu) return NAN;
  return ldexp(1.0, (int)(code & 0xFFu) - 127);
}

/* Round-to-nearest-even onto the E2M1 grid {0,.5,1,1.5,2,3,4,6}, saturating at
 * 6. Ties go to the code with mantissa bit 0 (the even code). */
unsigned orc_e2m1_encode(float x) {
  unsigned sign = signbit(x) ? 8u : 0u;
  double a = fabs((double)x);
  unsigned c;
  if (isnan(x)) return 7u; /* outside the contract: finite inputs only */
  for (c = 0; c < 7u; ++c) {
    double lo = orc_e2m1_value(c), hi = orc_e2m1_value(c + 1u);
    double mid = 0.5 * (lo + hi);
    if (a < mid) return sign | c;
    if (a == mid) return sign | ((c & 1u) ? c + 1u : c);
  }
  return sign | 7u;
}

/* Round-to-nearest-even onto the finite E4M3 values, saturating at 448
 * (infinities saturate too); NaN maps to 0x7F. Positive codes 0..126 are in
 * increasing order of value, so a bisection over codes finds the bracket. */
unsigned orc_e4m3_encode(float x) {
  unsigned sign = signbit(x) ? 0x80u : 0u;
  double a = fabs((double)x);
  unsigned lo = 0, hi = 126u, c;
  double vlo, vhi, mid;
  if (isnan(x)) return 0x7Fu;
  if (a >= 448.0) return sign | 0x7Eu;
  while (hi - lo > 1u) { /* invariant: value(lo) <= a < value(hi) */
    unsigned m = (lo + hi) / 2u;
    if (orc_e4m3_value(m) <= a) lo = m; else hi = m;
  }
  vlo = orc_e4m3_value(lo);
  vhi = orc_e4m3_value(hi);
  mid = 0.5 * (vlo + vhi);
  if (a < mid) c = lo;
  else if (a > mid) c = hi;
  else c = (lo & 1u) ? hi : lo;
  return sign | c;
}

static unsigned nibble(const uint8_t* row, int i) {
  return (i & 1) ? (unsigned)(row[i >> 1] >> 4) : (unsigned)(row[i >> 1] & 0xFu);
}

static void put_nibble(uint8_t* row, int i, unsigned code) {
  if (i & 1) row[i >> 1] = (uint8_t)((row[i >> 1] & 0x0Fu) | ((code & 0xFu) << 4));
  else       row[i >> 1] = (uint8_t)((row[i >> 1] & 0xF0u) | (code & 0xFu));
}

/* ------------------------------------------------------------------------ */
/* MXFP4 ([R] 2.4.4 OCP MXFP4; [B] 2: E2M1 values, one E8M0 per 32)          */
/* ------------------------------------------------------------------------ */

/* Shared exponent of one 32-element block: floor(log2(amax)) minus the
 * largest E2M1 exponent (2), clamped to the E8M0 range. */
static int mx_shared_exponent(const float* x) {
  float amax = 0.0f;
  int i, e, X;
  for (i = 0; i < ORC_MX_BLOCK; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  if (amax == 0.0f) return -127;
  (void)frexp((double)amax, &e); /* amax = f * 2^e, f in [0.5, 1) */
  X = (e - 1) - 2;
  if (X < -127) X = -127;
  if (X > 127) X = 127;
  return X;
}

void orc_quant_mxfp4(const float* x, int64_t rows, int cols, uint8_t* data,
                     uint8_t* e8m0) {
  int64_t r;
  int nb = cols / ORC_MX_BLOCK;
  /* rows are independent; OpenMP only spreads them over cores */
#ifdef _OPENMP
#pragma omp parallel for schedule(static) if (rows > 4096)
#endif
  for (r = 0; r < rows; ++r) {
    const float* xr = x + r * cols;
    uint8_t* dr = data + r * (cols / 2);
    int b, i;
    memset(dr, 0, (size_t)(cols / 2));
    for (b = 0; b < nb; ++b) {
      int X = mx_shared_exponent(xr + b * ORC_MX_BLOCK);
      e8m0[r * nb + b] = (uint8_t)(X + 127);
      for (i = 0; i < ORC_MX_BLOCK; ++i) {
        /* x * 2^-X: exact for every value that can round to a nonzero code */
        float v = (float)ldexp((double)xr[b * ORC_MX_BLOCK + i], -X);
        put_nibble(dr, b * ORC_MX_BLOCK + i, orc_e2m1_encode(v));
      }
    }
  }
}

void orc_dequant_mxfp4(const uint8_t* data, const uint8_t* e8m0, int64_t rows,
                       int cols, double* out) {
  int64_t r;
  int nb = cols / ORC_MX_BLOCK, c;
  for (r = 0; r < rows; ++r)
    for (c = 0; c < cols; ++c)
      out[r * cols + c] = orc_e2m1_value(nibble(data + r * (cols / 2), c)) *
                          orc_e8m0_value(e8m0[r * nb + c / ORC_MX_BLOCK]);
}

/* ------------------------------------------------------------------------ */
/* Main KV: E2M1 + one E4M3 scale per 16 channels, no global scale           */
/* ([R] 2.4.4; [B] 2 "4.5 bit per channel"; [B] 5)                           */
/* ------------------------------------------------------------------------ */

void orc_pack_kv_fp4(const float* x, int64_t n, uint8_t* kv_data,
                     uint8_t* kv_scale) {
  int64_t t;
  const int nb = ORC_KV_DIM / ORC_KV_BLOCK;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) if (n > 4096)
#endif
  for (t = 0; t < n; ++t) {
    const float* xr = x + t * ORC_KV_DIM;
    uint8_t* dr = kv_data + t * (ORC_KV_DIM / 2);
    int b, i;
    memset(dr, 0, ORC_KV_DIM / 2);
    for (b = 0; b < nb; ++b) {
      float amax = 0.0f, sf;
      unsigned sc;
      for (i = 0; i < ORC_KV_BLOCK; ++i) {
        float a = fabsf(xr[b * ORC_KV_BLOCK + i]);
        if (a > amax) amax = a;
      }
      sf = amax / 6.0f; /* IEEE fp32 quotient */
      sc = orc_e4m3_encode(sf);
      kv_scale[t * nb + b] = (uint8_t)sc;
      sf = (float)orc_e4m3_value(sc);
      for (i = 0; i < ORC_KV_BLOCK; ++i) {
        unsigned code = 0u;
        if (sf != 0.0f) code = orc_e2m1_encode(xr[b * ORC_KV_BLOCK + i] / sf);
        put_nibble(dr, b * ORC_KV_BLOCK + i, code);
      }
    }
  }
}

void orc_unpack_kv_fp4(const uint8_t* kv_data, const uint8_t* kv_scale,
                       int64_t n, double* out) {
  int64_t t;
  const int nb = ORC_KV_DIM / ORC_KV_BLOCK;
  int c;
  for (t = 0; t < n; ++t)
    for (c = 0; c < ORC_KV_DIM; ++c)
      out[t * ORC_KV_DIM + c] =
          orc_e2m1_value(nibble(kv_data + t * (ORC_KV_DIM / 2), c)) *
          orc_e4m3_value(kv_scale[t * nb + c / ORC_KV_BLOCK]);
}

/* SWA KV stays FP8 E4M3 ([R] 2.4.4 last paragraph); no scale is described. */
void orc_pack_fp8(const float* x, int64_t n, uint8_t* out) {
  int64_t i;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) if (n > 65536)
#endif
  for (i = 0; i < n; ++i) out[i] = (uint8_t)orc_e4m3_encode(x[i]);
}

void orc_unpack_fp8(const uint8_t* in, int64_t n, double* out) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = orc_e4m3_value(in[i]);
}

/* [B] 2: main KV 512 x 4 bit + 32 scale bytes; indexer K 64 + 4 bytes. */
int orc_main_kv_entry_bytes(void) {
  return ORC_KV_DIM / 2 + ORC_KV_DIM / ORC_KV_BLOCK;
}
int orc_indexer_k_entry_bytes(void) {
  return ORC_IDX_DIM / 2 + ORC_IDX_DIM / ORC_MX_BLOCK;
}

/* ------------------------------------------------------------------------ */
/* Lightning-indexer score ([R] 2.3 and 2.3.2; [B] 4.1 and 4.4)               */
/* ------------------------------------------------------------------------ */

uint64_t orc_index_score(const uint8_t* q_data, const uint8_t* q_e8m0,
                         const float* w, const uint8_t* ik_data,
                         const uint8_t* ik_scale, const int32_t* positions,
                         int64_t n, float* out32, double* out64) {
  double q[ORC_IDX_HEADS][ORC_IDX_DIM];
  uint64_t macs = 0;
  int64_t i;
  orc_dequant_mxfp4(q_data, q_e8m0, ORC_IDX_HEADS, ORC_IDX_DIM, &q[0][0]);
  /* entries are independent; OpenMP only spreads them over cores */
#ifdef _OPENMP
#pragma omp parallel for schedule(static) reduction(+ : macs) if (n > 8192)
#endif
  for (i = 0; i < n; ++i) {
    int64_t p = positions ? (int64_t)positions[i] : i;
    double s = 0.0, k[ORC_IDX_DIM];
    int h, c;
    if (p < 0) {
      out32[i] = -INFINITY;
      if (out64) out64[i] = -INFINITY;
      continue;
    }
    orc_dequant_mxfp4(ik_data + p * (ORC_IDX_DIM / 2),
                      ik_scale + p * (ORC_IDX_DIM / ORC_MX_BLOCK), 1,
                      ORC_IDX_DIM, k);
    for (h = 0; h < ORC_IDX_HEADS; ++h) {
      double dot = 0.0;
      for (c = 0; c < ORC_IDX_DIM; ++c) dot += q[h][c] * k[c];
      macs += ORC_IDX_DIM;
      s += (double)w[h] * (dot > 0.0 ? dot : 0.0);
    }
    out32[i] = (float)s;
    if (out64) out64[i] = s;
  }
  return macs;
}

/* ------------------------------------------------------------------------ */
/* Top-K ([R] 2.3 "selects the Top-K entries for each query"; K = 512 [B] 1)  */
/* ------------------------------------------------------------------------ */

typedef struct {
  float s;
  int32_t p;
} scored_t;

static int by_score_desc_pos_asc(const void* a, const void* b) {
  const scored_t* x = (const scored_t*)a;
  const scored_t* y = (const scored_t*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->p > y->p) - (x->p < y->p);
}

int orc_topk(const float* scores, const int32_t* positions, int64_t n, int k,
             int32_t* idx) {
  scored_t* v = (scored_t*)malloc(sizeof(scored_t) * (size_t)(n > 0 ? n : 1));
  int64_t i, m = 0;
  int j, out;
  for (i = 0; i < n; ++i) {
    int32_t p = positions ? positions[i] : (int32_t)i;
    if (p < 0 || isnan(scores[i]) || scores[i] == -INFINITY) continue;
    v[m].s = scores[i];
    v[m].p = p;
    ++m;
  }
  qsort(v, (size_t)m, sizeof(scored_t), by_score_desc_pos_asc);
  out = (int)(m < k ? m : k);
  for (j = 0; j < k; ++j) idx[j] = j < out ? v[j].p : -1;
  free(v);
  return out;
}

/* ------------------------------------------------------------------------ */
/* Hierarchical Sparse Indexer pool ([R] 2.3.2 and Figure 5; [B] 1, 4.3)      */
/* ------------------------------------------------------------------------ */

static int by_int_asc(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

void orc_block_max(const float* scores, int64_t n, int block, float* bmax) {
  int64_t nb = (n + block - 1) / block, b, p;
  for (b = 0; b < nb; ++b) {
    float m = -INFINITY;
    for (p = b * block; p < (b + 1) * block && p < n; ++p)
      if (scores[p] > m) m = scores[p];
    bmax[b] = m;
  }
}

int orc_block_pool(const float* scores, int64_t n, int block, int n_blocks,
                   int32_t* pool) {
  int64_t nb = (n + block - 1) / block, b;
  float* bmax = (float*)malloc(sizeof(float) * (size_t)(nb > 0 ? nb : 1));
  int32_t* kept = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_blocks > 0 ? n_blocks : 1));
  int j, r, n_kept;
  (void)b;
  orc_block_max(scores, n, block, bmax);
  /* the best blocks by (max desc, block asc) are a Top-K over block maxima */
  n_kept = orc_topk(bmax, NULL, nb, n_blocks, kept);
  qsort(kept, (size_t)n_kept, sizeof(int32_t), by_int_asc);
  for (j = 0; j < n_blocks; ++j)
    for (r = 0; r < block; ++r) {
      int64_t p = j < n_kept ? (int64_t)kept[j] * block + r : -1;
      pool[(int64_t)j * block + r] = (p >= 0 && p < n) ? (int32_t)p : -1;
    }
  free(bmax);
  free(kept);
  return n_kept;
}

/* ------------------------------------------------------------------------ */
/* Sparse attention over the selected latents plus the SWA window            */
/* ([R] 2.3: "each Q attends to the selected entries together with the       */
/* layer-local sliding-window KV"; [B] 1: 64 heads, head dim 512, the        */
/* 512-dim latent shared as K and V)                                         */
/* ------------------------------------------------------------------------ */

void orc_sparse_attn(const float* q, int H, int D, const uint8_t* kv_data,
                     const uint8_t* kv_scale, const int32_t* idx, int k,
                     const uint8_t* swa, int n_swa, double sm_scale,
                     double* out, double* lse) {
  int n_rows = 0, t, h, c;
  double* rows = (double*)malloc(sizeof(double) * (size_t)(k + n_swa + 1) * (size_t)D);
  double* s = (double*)malloc(sizeof(double) * (size_t)(k + n_swa + 1));
  for (t = 0; t < k; ++t) {
    if (idx[t] < 0) continue;
    orc_unpack_kv_fp4(kv_data + (int64_t)idx[t] * (D / 2),
                      kv_scale + (int64_t)idx[t] * (D / ORC_KV_BLOCK), 1,
                      rows + (int64_t)n_rows * D);
    ++n_rows;
  }
  for (t = 0; t < n_swa; ++t) {
    orc_unpack_fp8(swa + (int64_t)t * D, D, rows + (int64_t)n_rows * D);
    ++n_rows;
  }
  for (h = 0; h < H; ++h) {
    double m = -INFINITY, l = 0.0;
    for (t = 0; t < n_rows; ++t) {
      double dot = 0.0;
      for (c = 0; c < D; ++c) dot += (double)q[h * D + c] * rows[(int64_t)t * D + c];
      s[t] = sm_scale * dot;
      if (s[t] > m) m = s[t];
    }
    for (c = 0; c < D; ++c) out[h * D + c] = 0.0;
    if (n_rows == 0) {
      lse[h] = -INFINITY;
      continue;
    }
    for (t = 0; t < n_rows; ++t) {
      double p = exp(s[t] - m);
      l += p;
      for (c = 0; c < D; ++c) out[h * D + c] += p * rows[(int64_t)t * D + c];
    }
    for (c = 0; c < D; ++c) out[h * D + c] /= l;
    lse[h] = m + log(l);
  }
  free(rows);
  free(s);
}

/* ------------------------------------------------------------------------ */
/* A decode step for a batch: score -> Top-K -> attention for the indexing    */
/* layer and the Reuse layers that share its indices ([R] 2.3.1)              */
/* ------------------------------------------------------------------------ */

uint64_t orc_decode_batch(int B, int64_t cap, const int32_t* n_visible,
                          const uint8_t* q_data, const uint8_t* q_e8m0,
                          const float* w, const uint8_t* ik_data,
                          const uint8_t* ik_scale, const uint8_t* kv_data,
                          const uint8_t* kv_scale, int k, int L,
                          const float* Q, int H, int D, const uint8_t* swa,
                          int n_swa, double sm_scale, int32_t* idx,
                          double* out, int n_threads) {
  uint64_t macs = 0;
  int b;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : macs)
#endif
  for (b = 0; b < B; ++b) {
    int64_t n = n_visible[b];
    float* s = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
    double* lse = (double*)malloc(sizeof(double) * (size_t)H);
    int l;
    macs += orc_index_score(q_data + (int64_t)b * ORC_IDX_HEADS * (ORC_IDX_DIM / 2),
                            q_e8m0 + (int64_t)b * ORC_IDX_HEADS * (ORC_IDX_DIM / ORC_MX_BLOCK),
                            w + (int64_t)b * ORC_IDX_HEADS,
                            ik_data + (int64_t)b * cap * (ORC_IDX_DIM / 2),
                            ik_scale + (int64_t)b * cap * (ORC_IDX_DIM / ORC_MX_BLOCK),
                            NULL, n, s, NULL);
    orc_topk(s, NULL, n, k, idx + (int64_t)b * k);
    for (l = 0; l < L; ++l)
      orc_sparse_attn(Q + ((int64_t)b * L + l) * H * D, H, D,
                      kv_data + (int64_t)b * cap * (D / 2),
                      kv_scale + (int64_t)b * cap * (D / ORC_KV_BLOCK),
                      idx + (int64_t)b * k, k,
                      swa + ((int64_t)b * L + l) * n_swa * D, n_swa, sm_scale,
                      out + ((int64_t)b * L + l) * H * D, lse);
    free(s);
    free(lse);
  }
  (void)n_threads;
  return macs;
}

/* ------------------------------------------------------------------------ */
/* Attention over a union of disjoint row sets ([R] 2.3: one softmax over     */
/* all rows a query attends to, split here by where the rows live)           */
/* ------------------------------------------------------------------------ */

void orc_attn_merge(const double* outs, const double* lses, int R, int H,
                    int D, double* out, double* lse) {
  int r, h, c;
  for (h = 0; h < H; ++h) {
    double m = -INFINITY, l = 0.0;
    for (r = 0; r < R; ++r)
      if (lses[(int64_t)r * H + h] > m) m = lses[(int64_t)r * H + h];
    for (c = 0; c < D; ++c) out[(int64_t)h * D + c] = 0.0;
    if (m == -INFINITY) {
      lse[h] = -INFINITY;
      continue;
    }
    for (r = 0; r < R; ++r) l += exp(lses[(int64_t)r * H + h] - m);
    lse[h] = m + log(l);
    for (r = 0; r < R; ++r) {
      double wgt = exp(lses[(int64_t)r * H + h] - lse[h]);
      if (lses[(int64_t)r * H + h] == -INFINITY) continue;
      for (c = 0; c < D; ++c)
        out[(int64_t)h * D + c] += wgt * outs[((int64_t)r * H + h) * D + c];
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Sequence compressor ([V4] "Compressed Sparse Attention": m tokens merge    */
/* into one compressed entry by a softmax over the group; [B] 4.1: CSA2       */
/* blocks do not overlap)                                                    */
/* ------------------------------------------------------------------------ */

void orc_compress_kv(const double* C, const double* Z, const double* bias,
                     int64_t n_tokens, int m, int D, double* out) {
  int64_t e, n_out = n_tokens / m;
  int a, c;
  for (e = 0; e < n_out; ++e)
    for (c = 0; c < D; ++c) {
      double mx = -INFINITY, den = 0.0, num = 0.0;
      for (a = 0; a < m; ++a) {
        double s = Z[(e * m + a) * D + c] + bias[a * D + c];
        if (s > mx) mx = s;
      }
      for (a = 0; a < m; ++a) {
        double wgt = exp(Z[(e * m + a) * D + c] + bias[a * D + c] - mx);
        den += wgt;
        num += wgt * C[(e * m + a) * D + c];
      }
      out[e * D + c] = num / den;
    }
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
