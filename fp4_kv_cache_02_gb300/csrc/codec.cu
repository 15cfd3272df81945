// codec.cu -- FP4 / FP8 pack and unpack kernels.
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression",
// section 2.4.4: OCP MXFP4 for the indexer q/k (one E8M0 scale per 32, mer.dev
// notes section 2), E2M1 with one E4M3 scale per 16 channels and no global
// scale for the main KV, FP8 (E4M3) for the SWA KV.
//
// These kernels are memory bound and off the per-query hot loop except for
// the indexer-q quantisation; they use one thread per scale block with
// 16-byte vector loads. The fused KV append (a new entry's main-KV latent,
// quantised after RoPE, and its indexer key, written at the sequence's next
// position) uses one warp per entry and the same block encoders.
#include "codec_blocks.cuh"

namespace csa2 {

__device__ int g_codec_error = 0;

// ---- MXFP4: one thread per 32-element block ---------------------------------
__global__ void quant_mxfp4_kernel(const uint16_t* __restrict__ x, int64_t n_blocks,
                                   uint8_t* __restrict__ data, uint8_t* __restrict__ e8m0) {
  pdl_begin();
  int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (blk >= n_blocks) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + blk * 32);
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 v = src[i];
    w[4 * i + 0] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
  }
  uint4 d;
  uint8_t e;
  encode_mxfp4_block(w, d, e);
  *reinterpret_cast<uint4*>(data + blk * 16) = d;
  e8m0[blk] = e;
}

__global__ void dequant_mxfp4_kernel(const uint8_t* __restrict__ data,
                                     const uint8_t* __restrict__ e8m0, int64_t n_blocks,
                                     float* __restrict__ out) {
  int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (blk >= n_blocks) return;
  uint4 v = *reinterpret_cast<const uint4*>(data + blk * 16);
  float s = e8m0_to_f32(e8m0[blk]);
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float4* dst = reinterpret_cast<float4*>(out + blk * 32);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t b = w[i] >> (16 * j);
      dst[2 * i + j] = make_float4(e2m1_to_f32(b & 0xF) * s, e2m1_to_f32((b >> 4) & 0xF) * s,
                                   e2m1_to_f32((b >> 8) & 0xF) * s, e2m1_to_f32((b >> 12) & 0xF) * s);
    }
  }
}

// ---- main KV: one thread per 16-channel block ----------------------------------
__global__ void pack_kv_fp4_kernel(const uint16_t* __restrict__ x, int64_t n_blocks,
                                   uint8_t* __restrict__ kv_data, uint8_t* __restrict__ kv_scale) {
  int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (blk >= n_blocks) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + blk * 16);
  uint4 v0 = src[0], v1 = src[1];
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  uint2 d;
  uint8_t sc;
  encode_kv_fp4_block(w, d, sc);
  *reinterpret_cast<uint2*>(kv_data + blk * 8) = d;
  kv_scale[blk] = sc;
}

__global__ void unpack_kv_fp4_kernel(const uint8_t* __restrict__ kv_data,
                                     const uint8_t* __restrict__ kv_scale, int64_t n_blocks,
                                     uint16_t* __restrict__ out) {
  int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (blk >= n_blocks) return;
  uint2 v = *reinterpret_cast<const uint2*>(kv_data + blk * 8);
  float s = e4m3_to_f32(kv_scale[blk]);
  uint32_t w[2] = {v.x, v.y};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t b = (w[i] >> (8 * j)) & 0xFFu;
      // product of an E2M1 value and an E4M3 scale has <= 6 significant bits:
      // exact in bf16, so the round-to-nearest conversion is exact
      __nv_bfloat162 p = __floats2bfloat162_rn(e2m1_to_f32(b & 0xF) * s, e2m1_to_f32(b >> 4) * s);
      o[4 * i + j] = *reinterpret_cast<uint32_t*>(&p);
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(out + blk * 16);
  dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// ---- FP8 E4M3: one thread per 8 elements (tail handled elementwise) -------------
__global__ void pack_fp8_kernel(const uint16_t* __restrict__ x, int64_t n, uint8_t* __restrict__ out) {
  int64_t i8 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (i8 >= n) return;
  if (i8 + 8 <= n && ((((uintptr_t)(x + i8)) & 15) == 0) && ((((uintptr_t)(out + i8)) & 7) == 0)) {
    uint4 v = *reinterpret_cast<const uint4*>(x + i8);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t r0 = cvt_e4m3x2(bf16_bits_to_f32(w[0] & 0xFFFF), bf16_bits_to_f32(w[0] >> 16)) |
                  (cvt_e4m3x2(bf16_bits_to_f32(w[1] & 0xFFFF), bf16_bits_to_f32(w[1] >> 16)) << 16);
    uint32_t r1 = cvt_e4m3x2(bf16_bits_to_f32(w[2] & 0xFFFF), bf16_bits_to_f32(w[2] >> 16)) |
                  (cvt_e4m3x2(bf16_bits_to_f32(w[3] & 0xFFFF), bf16_bits_to_f32(w[3] >> 16)) << 16);
    *reinterpret_cast<uint2*>(out + i8) = make_uint2(r0, r1);
  } else {
    for (int64_t i = i8; i < n && i < i8 + 8; ++i)
      out[i] = (uint8_t)(cvt_e4m3x2(bf16_bits_to_f32(x[i]), 0.0f) & 0xFF);
  }
}

__global__ void unpack_fp8_kernel(const uint8_t* __restrict__ in, int64_t n, uint16_t* __restrict__ out) {
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  __nv_bfloat16 b = __float2bfloat16_rn(e4m3_to_f32(in[i]));
  out[i] = *reinterpret_cast<uint16_t*>(&b);
}

// ---- fused append: one warp per kPerWarp new entries (b, t) ------------------
// The warp issues all its entries' loads before encoding any (two entries a
// warp for bulk appends; one for small batches, where the grid is the limit).
// Lane l encodes
// main-KV block l (channels 16l .. 16l+15) and indexer-key channels 4l .. 4l+3:
// the eight lanes of an MXFP4 block (32 channels) share its amax through
// shuffles. An entry goes to position n_visible[b] + t. A sequence whose T
// entries do not fit below the capacity (or whose count is negative) gets
// none of them, keeps its count and records a device error.
constexpr int kAppendWarps = 8;
constexpr int64_t kAppendPairsFrom = 16384;  // entries from which a warp takes two

template <int kPerWarp>
__global__ void __launch_bounds__(kAppendWarps * 32) kv_append_kernel(
    const uint16_t* __restrict__ kv, const uint16_t* __restrict__ ik, int32_t B, int32_t T,
    uint8_t* __restrict__ kv_data, uint8_t* __restrict__ kv_scale, uint8_t* __restrict__ ik_data,
    uint8_t* __restrict__ ik_scale, int64_t cap, const int32_t* __restrict__ n_visible,
    int32_t* __restrict__ n_visible_out) {
  static_assert(kIdxDim == 32 * 4 && kHeadDim == 32 * 16, "a lane holds 16 latent and 4 key channels");
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int64_t entries = (int64_t)B * T;
  const int64_t e0 = ((int64_t)blockIdx.x * kAppendWarps + (threadIdx.x >> 5)) * kPerWarp;
  if (e0 >= entries) return;
  uint4 kv_lo[kPerWarp], kv_hi[kPerWarp];
  uint2 ikw[kPerWarp];
  int64_t nvs[kPerWarp];
  int bs[kPerWarp], ts[kPerWarp];
#pragma unroll
  for (int j = 0; j < kPerWarp; ++j) {
    const int64_t e = e0 + j;
    if (e < entries) {
      const uint4* src = reinterpret_cast<const uint4*>(kv + e * kHeadDim + lane * 16);
      kv_lo[j] = src[0];
      kv_hi[j] = src[1];
      ikw[j] = reinterpret_cast<const uint2*>(ik + e * kIdxDim)[lane];
      // (a 32-bit division whenever the entry index fits)
      bs[j] = e <= 0x7FFFFFFF ? (int)((uint32_t)e / (uint32_t)T) : (int)(e / T);
      ts[j] = (int)(e - (int64_t)bs[j] * T);
      nvs[j] = n_visible[bs[j]];
    }
  }
#pragma unroll
  for (int j = 0; j < kPerWarp; ++j) {
    const int64_t e = e0 + j;
    if (e >= entries) break;
    const int b = bs[j], t = ts[j];
    const int64_t nv = nvs[j];
    const bool fits = nv >= 0 && nv + T <= cap;
    if (n_visible_out && t == 0 && lane == 0) n_visible_out[b] = (int32_t)(fits ? nv + T : nv);
    if (!fits) {
      if (lane == 0 && t == 0) record_error(&g_codec_error, CSA2_ERR_DEVICE);
      continue;
    }
    const int64_t row = (int64_t)b * cap + nv + t;
    {
      const uint32_t w[8] = {kv_lo[j].x, kv_lo[j].y, kv_lo[j].z, kv_lo[j].w,
                             kv_hi[j].x, kv_hi[j].y, kv_hi[j].z, kv_hi[j].w};
      uint2 d;
      uint8_t sc;
      encode_kv_fp4_block(w, d, sc);
      *reinterpret_cast<uint2*>(kv_data + row * kKvBytes + lane * 8) = d;
      kv_scale[row * kKvScales + lane] = sc;
    }
    {
      uint32_t amax_bits = max(max(ikw[j].x & 0x7FFFu, (ikw[j].x >> 16) & 0x7FFFu),
                               max(ikw[j].y & 0x7FFFu, (ikw[j].y >> 16) & 0x7FFFu));
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) amax_bits = max(amax_bits, __shfl_xor_sync(0xffffffffu, amax_bits, o));
      float inv;
      const int X = mxfp4_exponent(amax_bits, inv);
      *reinterpret_cast<uint16_t*>(ik_data + row * (kIdxDim / 2) + lane * 2) =
          (uint16_t)encode_e2m1x4(ikw[j].x, ikw[j].y, inv);
      if ((lane & 7) == 0) ik_scale[row * (kIdxDim / 32) + lane / 8] = (uint8_t)(X + 127);
    }
  }
}

// ---- compressor: one warp per compressed entry --------------------------------
// entry e of m tokens (rows em .. em+m-1): per channel c the weights are a
// softmax over the block's tokens of Z[row][c] + bias[a][c], and the entry is
// the weighted sum of C[row][c]; it is rounded to bf16 and packed like the
// latent of csa2_kv_append. Lane l owns channels 16l .. 16l+15 (one E4M3 block).
// kM > 0 fixes m at compile time: every load of the entry (Z, C and the bias
// rows) is issued before the arithmetic. kM = 0 walks a runtime m. Both do the
// same operations in the same order, so they give the same bits.
template <int kM>
__global__ void __launch_bounds__(kAppendWarps * 32) compress_kv_kernel(
    const uint16_t* __restrict__ C, const uint16_t* __restrict__ Z, const float* __restrict__ bias, int64_t n_out,
    int32_t m_rt, uint8_t* __restrict__ kv_data, uint8_t* __restrict__ kv_scale, uint16_t* __restrict__ out_bf16) {
  pdl_begin();
  const int m = kM > 0 ? kM : m_rt;
  const int lane = threadIdx.x & 31;
  const int64_t e = (int64_t)blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
  if (e >= n_out) return;
  const int c0 = lane * 16;
  auto load_words = [&](const uint16_t* base, int64_t row, uint32_t (&w)[8]) {
    const uint4* src = reinterpret_cast<const uint4*>(base + row * kHeadDim + c0);
    const uint4 a = src[0], b = src[1];
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  };
  auto load_bias = [&](int a, float (&v)[16]) {
    const float4* src = reinterpret_cast<const float4*>(bias + (int64_t)a * kHeadDim + c0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 x = src[q];
      v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
    }
  };
  auto lo = [](uint32_t w) { return bf16_bits_to_f32(w & 0xFFFFu); };
  auto hi = [](uint32_t w) { return bf16_bits_to_f32(w >> 16); };
  float mx[16], den[16], num[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) mx[i] = -INFINITY;
  if constexpr (kM > 0) {
    uint32_t zw[kM][8], cw[kM][8];
    float bv[kM][16];
#pragma unroll
    for (int a = 0; a < kM; ++a) {
      load_words(Z, e * kM + a, zw[a]);
      load_words(C, e * kM + a, cw[a]);
      load_bias(a, bv[a]);
    }
#pragma unroll
    for (int a = 0; a < kM; ++a)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        mx[2 * i] = fmaxf(mx[2 * i], lo(zw[a][i]) + bv[a][2 * i]);
        mx[2 * i + 1] = fmaxf(mx[2 * i + 1], hi(zw[a][i]) + bv[a][2 * i + 1]);
      }
#pragma unroll
    for (int i = 0; i < 16; ++i) den[i] = num[i] = 0.0f;
#pragma unroll
    for (int a = 0; a < kM; ++a)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float w0 = expf(lo(zw[a][i]) + bv[a][2 * i] - mx[2 * i]);
        const float w1 = expf(hi(zw[a][i]) + bv[a][2 * i + 1] - mx[2 * i + 1]);
        den[2 * i] += w0;
        den[2 * i + 1] += w1;
        num[2 * i] = fmaf(w0, lo(cw[a][i]), num[2 * i]);
        num[2 * i + 1] = fmaf(w1, hi(cw[a][i]), num[2 * i + 1]);
      }
  } else {
    uint32_t zw[8], cw[8];
    float bv[16];
    for (int a = 0; a < m; ++a) {
      load_words(Z, e * m + a, zw);
      load_bias(a, bv);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        mx[2 * i] = fmaxf(mx[2 * i], lo(zw[i]) + bv[2 * i]);
        mx[2 * i + 1] = fmaxf(mx[2 * i + 1], hi(zw[i]) + bv[2 * i + 1]);
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) den[i] = num[i] = 0.0f;
    for (int a = 0; a < m; ++a) {
      load_words(Z, e * m + a, zw);
      load_words(C, e * m + a, cw);
      load_bias(a, bv);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float w0 = expf(lo(zw[i]) + bv[2 * i] - mx[2 * i]);
        const float w1 = expf(hi(zw[i]) + bv[2 * i + 1] - mx[2 * i + 1]);
        den[2 * i] += w0;
        den[2 * i + 1] += w1;
        num[2 * i] = fmaf(w0, lo(cw[i]), num[2 * i]);
        num[2 * i + 1] = fmaf(w1, hi(cw[i]), num[2 * i + 1]);
      }
    }
  }
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(num[2 * i] / den[2 * i], num[2 * i + 1] / den[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
  if (out_bf16) {
    uint4* dst = reinterpret_cast<uint4*>(out_bf16 + e * kHeadDim + c0);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
  uint2 d;
  uint8_t sc;
  encode_kv_fp4_block(w, d, sc);
  *reinterpret_cast<uint2*>(kv_data + e * kKvBytes + lane * 8) = d;
  kv_scale[e * kKvScales + lane] = sc;
}

// In-place advance of the visible counts, after the append grid has finished
// reading them (its programmatic dependency waits for the whole grid).
__global__ void advance_visible_kernel(int32_t* __restrict__ n_visible, int32_t B, int32_t T, int64_t cap) {
  pdl_begin();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int64_t nv = n_visible[b];
  if (nv >= 0 && nv + T <= cap) n_visible[b] = (int32_t)(nv + T);
}

}  // namespace csa2

using namespace csa2;

static inline unsigned grid_for(int64_t n, int threads) {
  return (unsigned)((n + threads - 1) / threads);
}

int csa2_read_and_clear_codec_error(cudaStream_t s) {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_codec_error, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return CSA2_ERR_CUDA;
  if (cudaMemcpyToSymbolAsync(g_codec_error, &z, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return CSA2_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return CSA2_ERR_CUDA;
  return v;
}

extern "C" int csa2_quant_mxfp4(const void* x_bf16, int64_t rows, int32_t cols, uint8_t* data,
                                uint8_t* e8m0, csa2_stream_t stream) {
  if (!x_bf16 || !data || !e8m0 || rows < 0 || cols <= 0) return CSA2_ERR_INVALID_ARG;
  if (cols % 32) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (!csa2_aligned(x_bf16, 16) || !csa2_aligned(data, 16)) return CSA2_ERR_ALIGNMENT;
  int64_t nb = rows * (cols / 32);
  if (nb == 0) return CSA2_OK;
  CSA2_LAUNCH_PDL(quant_mxfp4_kernel, grid_for(nb, 256), dim3(256), 0, (cudaStream_t)stream,
                  (const uint16_t*)x_bf16, nb, data, e8m0);
  return CSA2_OK;
}

extern "C" int csa2_dequant_mxfp4(const uint8_t* data, const uint8_t* e8m0, int64_t rows, int32_t cols,
                                  float* out, csa2_stream_t stream) {
  if (!data || !e8m0 || !out || rows < 0 || cols <= 0) return CSA2_ERR_INVALID_ARG;
  if (cols % 32) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (!csa2_aligned(data, 16) || !csa2_aligned(out, 16)) return CSA2_ERR_ALIGNMENT;
  int64_t nb = rows * (cols / 32);
  if (nb == 0) return CSA2_OK;
  dequant_mxfp4_kernel<<<grid_for(nb, 256), 256, 0, (cudaStream_t)stream>>>(data, e8m0, nb, out);
  CSA2_CHECK_LAUNCH();
  return CSA2_OK;
}

extern "C" int csa2_pack_kv_fp4(const void* x_bf16, int64_t n, uint8_t* kv_data, uint8_t* kv_scale,
                                csa2_stream_t stream) {
  if (!x_bf16 || !kv_data || !kv_scale || n < 0) return CSA2_ERR_INVALID_ARG;
  if (!csa2_aligned(x_bf16, 16) || !csa2_aligned(kv_data, 8)) return CSA2_ERR_ALIGNMENT;
  int64_t nb = n * (kHeadDim / 16);
  if (nb == 0) return CSA2_OK;
  pack_kv_fp4_kernel<<<grid_for(nb, 256), 256, 0, (cudaStream_t)stream>>>(
      (const uint16_t*)x_bf16, nb, kv_data, kv_scale);
  CSA2_CHECK_LAUNCH();
  return CSA2_OK;
}

extern "C" int csa2_unpack_kv_fp4(const uint8_t* kv_data, const uint8_t* kv_scale, int64_t n,
                                  void* out_bf16, csa2_stream_t stream) {
  if (!kv_data || !kv_scale || !out_bf16 || n < 0) return CSA2_ERR_INVALID_ARG;
  if (!csa2_aligned(kv_data, 8) || !csa2_aligned(out_bf16, 16)) return CSA2_ERR_ALIGNMENT;
  int64_t nb = n * (kHeadDim / 16);
  if (nb == 0) return CSA2_OK;
  unpack_kv_fp4_kernel<<<grid_for(nb, 256), 256, 0, (cudaStream_t)stream>>>(
      kv_data, kv_scale, nb, (uint16_t*)out_bf16);
  CSA2_CHECK_LAUNCH();
  return CSA2_OK;
}

extern "C" int csa2_pack_fp8_e4m3(const void* x_bf16, int64_t n, uint8_t* out, csa2_stream_t stream) {
  if (!x_bf16 || !out || n < 0) return CSA2_ERR_INVALID_ARG;
  if (!csa2_aligned(x_bf16, 2)) return CSA2_ERR_ALIGNMENT;
  if (n == 0) return CSA2_OK;
  pack_fp8_kernel<<<grid_for((n + 7) / 8, 256), 256, 0, (cudaStream_t)stream>>>(
      (const uint16_t*)x_bf16, n, out);
  CSA2_CHECK_LAUNCH();
  return CSA2_OK;
}

extern "C" int csa2_unpack_fp8_e4m3(const uint8_t* in, int64_t n, void* out_bf16, csa2_stream_t stream) {
  if (!in || !out_bf16 || n < 0) return CSA2_ERR_INVALID_ARG;
  if (!csa2_aligned(out_bf16, 2)) return CSA2_ERR_ALIGNMENT;
  if (n == 0) return CSA2_OK;
  unpack_fp8_kernel<<<grid_for(n, 256), 256, 0, (cudaStream_t)stream>>>(in, n, (uint16_t*)out_bf16);
  CSA2_CHECK_LAUNCH();
  return CSA2_OK;
}

extern "C" int csa2_kv_append(const void* kv_bf16, const void* ik_bf16, int32_t B, int32_t T, uint8_t* kv_data,
                              uint8_t* kv_scale, uint8_t* ik_data, uint8_t* ik_scale, int64_t cap,
                              const int32_t* n_visible, int32_t* n_visible_out, csa2_stream_t stream) {
  if (!kv_bf16 || !ik_bf16 || !kv_data || !kv_scale || !ik_data || !ik_scale || !n_visible) return CSA2_ERR_INVALID_ARG;
  if (B < 0 || T < 0 || cap < 0) return CSA2_ERR_INVALID_ARG;
  if (cap > 0x7FFFFFFFLL) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (!csa2_aligned(kv_bf16, 16) || !csa2_aligned(ik_bf16, 16) || !csa2_aligned(kv_data, 8) ||
      !csa2_aligned(ik_data, 16))
    return CSA2_ERR_ALIGNMENT;
  if (B == 0 || T == 0) return CSA2_OK;
  cudaStream_t s = (cudaStream_t)stream;
  const bool in_place = n_visible_out == n_visible;
  const int64_t entries = (int64_t)B * T;
  int32_t* nv_out = in_place ? (int32_t*)nullptr : n_visible_out;
  if (entries >= kAppendPairsFrom)
    CSA2_LAUNCH_PDL(kv_append_kernel<2>, grid_for((entries + 1) / 2, kAppendWarps), dim3(kAppendWarps * 32), 0, s,
                    (const uint16_t*)kv_bf16, (const uint16_t*)ik_bf16, B, T, kv_data, kv_scale, ik_data, ik_scale,
                    cap, n_visible, nv_out);
  else
    CSA2_LAUNCH_PDL(kv_append_kernel<1>, grid_for(entries, kAppendWarps), dim3(kAppendWarps * 32), 0, s,
                    (const uint16_t*)kv_bf16, (const uint16_t*)ik_bf16, B, T, kv_data, kv_scale, ik_data, ik_scale,
                    cap, n_visible, nv_out);
  if (in_place)
    CSA2_LAUNCH_PDL(advance_visible_kernel, grid_for(B, 256), dim3(256), 0, s, n_visible_out, B, T, cap);
  return CSA2_OK;
}

extern "C" int csa2_compress_kv(const void* c_bf16, const void* z_bf16, const float* bias, int64_t n_tokens,
                                int32_t m, uint8_t* kv_data, uint8_t* kv_scale, void* out_bf16,
                                csa2_stream_t stream) {
  if (!c_bf16 || !z_bf16 || !bias || !kv_data || !kv_scale || n_tokens < 0 || m < 1) return CSA2_ERR_INVALID_ARG;
  if (n_tokens % m) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (!csa2_aligned(c_bf16, 16) || !csa2_aligned(z_bf16, 16) || !csa2_aligned(bias, 16) ||
      !csa2_aligned(kv_data, 8) || (out_bf16 && !csa2_aligned(out_bf16, 16)))
    return CSA2_ERR_ALIGNMENT;
  const int64_t n_out = n_tokens / m;
  if (n_out == 0) return CSA2_OK;
  const dim3 grid(grid_for(n_out, kAppendWarps)), block(kAppendWarps * 32);
  cudaStream_t s = (cudaStream_t)stream;
  const uint16_t *cp = (const uint16_t*)c_bf16, *zp = (const uint16_t*)z_bf16;
  if (m == 1)
    CSA2_LAUNCH_PDL(compress_kv_kernel<1>, grid, block, 0, s, cp, zp, bias, n_out, m, kv_data, kv_scale,
                    (uint16_t*)out_bf16);
  else if (m == 2)
    CSA2_LAUNCH_PDL(compress_kv_kernel<2>, grid, block, 0, s, cp, zp, bias, n_out, m, kv_data, kv_scale,
                    (uint16_t*)out_bf16);
  else
    CSA2_LAUNCH_PDL(compress_kv_kernel<0>, grid, block, 0, s, cp, zp, bias, n_out, m, kv_data, kv_scale,
                    (uint16_t*)out_bf16);
  return CSA2_OK;
}
