// codec.cu -- FP4 / FP8 pack and unpack kernels.
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression",
// section 2.4.4: OCP MXFP4 for the indexer q/k (one E8M0 scale per 32, mer.dev
// notes section 2), E2M1 with one E4M3 scale per 16 channels and no global
// scale for the main KV, FP8 (E4M3) for the SWA KV.
//
// These kernels are memory bound and off the per-query hot loop except for
// the indexer-q quantisation; they use one thread per scale block with
// 16-byte vector loads.
#include "common.cuh"

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
  // amax over the block, on the bf16 bit patterns with the sign cleared
  uint32_t amax_bits = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    amax_bits = max(amax_bits, (w[i] & 0x7FFFu));
    amax_bits = max(amax_bits, ((w[i] >> 16) & 0x7FFFu));
  }
  // floor(log2(amax)) is the unbiased exponent field for a normal amax;
  // subnormal or zero amax clamps to -127.
  int exp_field = (int)(amax_bits >> 7);  // bf16 exponent field
  int X = exp_field == 0 ? -127 : (exp_field - 127) - 2;
  X = X < -127 ? -127 : (X > 127 ? 127 : X);
  // 2^-X as fp32 (X = 127 gives the subnormal 2^-127)
  float inv = X == 127 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)(127 - X) << 23);
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t pair0 = w[4 * i + 2 * j], pair1 = w[4 * i + 2 * j + 1];
      float a0 = bf16_bits_to_f32(pair0 & 0xFFFFu) * inv;
      float a1 = bf16_bits_to_f32(pair0 >> 16) * inv;
      float a2 = bf16_bits_to_f32(pair1 & 0xFFFFu) * inv;
      float a3 = bf16_bits_to_f32(pair1 >> 16) * inv;
      word |= (cvt_e2m1x2(a0, a1) | (cvt_e2m1x2(a2, a3) << 8)) << (16 * j);
    }
    out[i] = word;
  }
  *reinterpret_cast<uint4*>(data + blk * 16) = make_uint4(out[0], out[1], out[2], out[3]);
  e8m0[blk] = (uint8_t)(X + 127);
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
  uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  float f[16];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
    f[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
    amax = fmaxf(amax, fabsf(f[2 * i]));
    amax = fmaxf(amax, fabsf(f[2 * i + 1]));
  }
  float q = __fdiv_rn(amax, 6.0f);
  uint32_t sc = cvt_e4m3x2(q, 0.0f) & 0xFFu;
  float s = e4m3_to_f32(sc);
  uint32_t out0 = 0, out1 = 0;
  if (s != 0.0f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t byte = cvt_e2m1x2(__fdiv_rn(f[2 * i], s), __fdiv_rn(f[2 * i + 1], s));
      out0 |= byte << (8 * i);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t byte = cvt_e2m1x2(__fdiv_rn(f[8 + 2 * i], s), __fdiv_rn(f[8 + 2 * i + 1], s));
      out1 |= byte << (8 * i);
    }
  }
  *reinterpret_cast<uint2*>(kv_data + blk * 8) = make_uint2(out0, out1);
  kv_scale[blk] = (uint8_t)sc;
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
