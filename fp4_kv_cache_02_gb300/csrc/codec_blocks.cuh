// codec_blocks.cuh -- encoders of one scale block, shared by the pack kernels
// and the fused KV append so that both write identical bytes.
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression",
// section 2.4.4: OCP MXFP4 (E2M1 values, one E8M0 scale per 32) for the
// indexer keys and queries; E2M1 with one E4M3 scale per 16 channels and no
// global scale for the main KV latent.
#pragma once
#include "common.cuh"

namespace csa2 {

// One MXFP4 block: 32 bf16 values (16 words of bf16 pairs, element 2i in the
// low half) -> 16 bytes of E2M1 pairs (element 2i in the low nibble) and the
// E8M0 code. The shared exponent is floor(log2(amax)) - 2 (the largest E2M1
// magnitude is 6 = 1.5 * 2^2), clamped to the E8M0 range; values are scaled
// by its power of two and rounded to nearest-even E2M1, saturating.
// The shared exponent X of an MXFP4 block, from the largest magnitude bit
// pattern (sign cleared) among its bf16 values, and the scaling 2^-X as fp32.
__device__ __forceinline__ int mxfp4_exponent(uint32_t amax_bits, float& inv) {
  // floor(log2(amax)) is the unbiased exponent field for a normal amax;
  // subnormal or zero amax clamps to -127.
  const int exp_field = (int)(amax_bits >> 7);  // bf16 exponent field
  int X = exp_field == 0 ? -127 : (exp_field - 127) - 2;
  X = X < -127 ? -127 : (X > 127 ? 127 : X);
  // 2^-X as fp32 (X = 127 gives the subnormal 2^-127)
  inv = X == 127 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)(127 - X) << 23);
  return X;
}

// Four consecutive values of an MXFP4 block (two words of bf16 pairs), scaled
// by 2^-X and rounded to nearest-even E2M1, saturating: two bytes, element 0 in
// the low nibble.
__device__ __forceinline__ uint32_t encode_e2m1x4(uint32_t pair0, uint32_t pair1, float inv) {
  const float a0 = bf16_bits_to_f32(pair0 & 0xFFFFu) * inv;
  const float a1 = bf16_bits_to_f32(pair0 >> 16) * inv;
  const float a2 = bf16_bits_to_f32(pair1 & 0xFFFFu) * inv;
  const float a3 = bf16_bits_to_f32(pair1 >> 16) * inv;
  return cvt_e2m1x2(a0, a1) | (cvt_e2m1x2(a2, a3) << 8);
}

__device__ __forceinline__ void encode_mxfp4_block(const uint32_t (&w)[16], uint4& data, uint8_t& e8m0) {
  uint32_t amax_bits = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    amax_bits = max(amax_bits, (w[i] & 0x7FFFu));
    amax_bits = max(amax_bits, ((w[i] >> 16) & 0x7FFFu));
  }
  float inv;
  const int X = mxfp4_exponent(amax_bits, inv);
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    out[i] = encode_e2m1x4(w[4 * i], w[4 * i + 1], inv) | (encode_e2m1x4(w[4 * i + 2], w[4 * i + 3], inv) << 16);
  data = make_uint4(out[0], out[1], out[2], out[3]);
  e8m0 = (uint8_t)(X + 127);
}

// One main-KV block: 16 bf16 values (8 words) -> 8 bytes of E2M1 pairs and
// the E4M3 scale. The scale is amax / 6 rounded to nearest-even E4M3 (6 is
// the largest E2M1 magnitude); each value is divided by the decoded scale and
// rounded to nearest-even E2M1, saturating. A zero scale stores zero codes.
__device__ __forceinline__ void encode_kv_fp4_block(const uint32_t (&w)[8], uint2& data, uint8_t& scale) {
  float f[16];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
    f[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
    amax = fmaxf(amax, fabsf(f[2 * i]));
    amax = fmaxf(amax, fabsf(f[2 * i + 1]));
  }
  const float q = __fdiv_rn(amax, 6.0f);
  const uint32_t sc = cvt_e4m3x2(q, 0.0f) & 0xFFu;
  const float s = e4m3_to_f32(sc);
  uint32_t out0 = 0, out1 = 0;
  if (s != 0.0f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out0 |= cvt_e2m1x2(__fdiv_rn(f[2 * i], s), __fdiv_rn(f[2 * i + 1], s)) << (8 * i);
      out1 |= cvt_e2m1x2(__fdiv_rn(f[8 + 2 * i], s), __fdiv_rn(f[8 + 2 * i + 1], s)) << (8 * i);
    }
  }
  data = make_uint2(out0, out1);
  scale = (uint8_t)sc;
}

}  // namespace csa2
