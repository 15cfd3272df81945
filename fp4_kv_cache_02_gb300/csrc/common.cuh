// common.cuh -- helpers shared by the CSA2 kernels (sm_103a).
//
// Format decoders here are written from the element-format definitions
// (E2M1: 1 sign, 2 exponent bits with bias 1, 1 mantissa bit; E4M3: bias 7,
// no infinity, S.1111.111 NaN; E8M0: bare exponent with bias 127), as used by
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" section
// 2.4.4 (OCP MXFP4 indexer q/k; E2M1 + E4M3-per-16 main KV; FP8 SWA KV).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/csa2.h"

namespace csa2 {

constexpr int kIdxHeads = CSA2_IDX_HEADS;  // 32
constexpr int kIdxDim = CSA2_IDX_DIM;      // 128
constexpr int kHeads = CSA2_HEADS;         // 64
constexpr int kHeadDim = CSA2_HEAD_DIM;    // 512
constexpr int kIkBytes = kIdxDim / 2;      // 64
constexpr int kIkScales = kIdxDim / 32;    // 4
constexpr int kKvBytes = kHeadDim / 2;     // 256
constexpr int kKvScales = kHeadDim / 16;   // 32
// Top-K histogram: bins are the top kTopkHistBits bits of score_key()
constexpr int kTopkHistBits = 12;
constexpr int kTopkHistBins = 1 << kTopkHistBits;

// ---- sticky device error word --------------------------------------------
// Each translation unit keeps its own word; csa2_get_last_error() collects
// them through the per-unit read_and_clear_* functions.
__device__ __forceinline__ void record_error(int* word, int status) {
  atomicCAS(word, 0, status);
}

// ---- element decoders ------------------------------------------------------
// E2M1 magnitude of a 4-bit code, as fp32.
__device__ __forceinline__ float e2m1_to_f32(uint32_t code) {
  uint32_t e = (code >> 1) & 3u, m = code & 1u;
  // normal: (1 + m/2) * 2^(e-1) -> fp32 bits exponent e-1+127, mantissa m<<22
  uint32_t normal = ((e + 126u) << 23) | (m << 22);
  float mag = e ? __uint_as_float(normal) : 0.5f * (float)m;
  return (code & 8u) ? -mag : mag;
}

// E4M3 value of an 8-bit code, as fp32 (NaN for 0x7F / 0xFF).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  uint32_t e = (code >> 3) & 15u, m = code & 7u;
  float mag;
  if (e == 15u && m == 7u) return __uint_as_float(0x7fc00000u);
  if (e) mag = __uint_as_float(((e + 120u) << 23) | (m << 20));
  else mag = (float)m * 0.001953125f;  // m * 2^-9
  return (code & 0x80u) ? -mag : mag;
}

// E8M0 scale 2^(code-127) as fp32 (code 0 -> 2^-127 is an fp32 subnormal).
__device__ __forceinline__ float e8m0_to_f32(uint32_t code) {
  if (code == 255u) return __uint_as_float(0x7fc00000u);
  if (code == 0u) return __uint_as_float(0x00400000u);  // 2^-127
  return __uint_as_float(code << 23);
}

// ---- encoders (hardware conversions, round-to-nearest-even, satfinite) ----
// Two fp32 values -> one byte of two E2M1 codes: `lo` in bits 0..3.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r) : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// Two fp32 values -> two E4M3 bytes: `lo` in bits 0..7.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---- order-preserving key of an fp32 score ---------------------------------
// Larger float -> larger unsigned key; -inf and NaN are not candidates.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t b = __float_as_uint(s);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ bool score_is_candidate(float s) {
  return !(isnan(s) || s == -INFINITY);
}

// ---- programmatic dependent launch ------------------------------------------
// The kernels of the decode chain begin here: wait until the kernel before this
// one in the stream has completed and its writes are visible, then allow the
// next kernel's CTAs to be scheduled (they park at their own wait). Launched
// without the programmatic-serialization attribute, both are no-ops.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// The two halves of pdl_begin() for kernels with a prologue that touches no
// memory the preceding kernel writes: let dependents launch now, wait later.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

}  // namespace csa2

// ---- host-side helpers -------------------------------------------------------
#define CSA2_CHECK_LAUNCH()                                 \
  do {                                                      \
    if (cudaPeekAtLastError() != cudaSuccess) {             \
      (void)cudaGetLastError();                             \
      return CSA2_ERR_CUDA;                                 \
    }                                                       \
  } while (0)

// Launches a kernel that begins with pdl_begin() so that its launch overlaps the
// tail of the previous kernel in the stream. Returns the launch status.
template <typename... KArgs, typename... Args>
static inline cudaError_t csa2_launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                          cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same with thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
static inline cudaError_t csa2_launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                                  cudaStream_t stream, unsigned cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

#define CSA2_LAUNCH_PDL(...)                                 \
  do {                                                      \
    if (csa2_launch_pdl(__VA_ARGS__) != cudaSuccess) {      \
      (void)cudaGetLastError();                             \
      return CSA2_ERR_CUDA;                                 \
    }                                                       \
  } while (0)

// Per-device "done" flags of one one-time set-up step, with the lock that
// orders the first calls of several host threads.
struct Csa2PerDeviceOnce {
  static constexpr int kMaxDevices = 64;
  std::mutex mu;
  bool done[kMaxDevices] = {};
};

// Opts `kernel` into `bytes` of dynamic shared memory on the current device,
// once per device (the attribute is per device; a kernel launched on a device
// where it was never set fails to launch above 48 KB).
static inline int csa2_smem_optin(const void* kernel, int bytes, Csa2PerDeviceOnce& once) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= Csa2PerDeviceOnce::kMaxDevices) return CSA2_ERR_CUDA;
  std::lock_guard<std::mutex> lock(once.mu);
  if (!once.done[dev]) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
      (void)cudaGetLastError();
      return CSA2_ERR_CUDA;
    }
    once.done[dev] = true;
  }
  return CSA2_OK;
}

static inline bool csa2_aligned(const void* p, uintptr_t a) {
  return (((uintptr_t)p) & (a - 1)) == 0;
}

// per-translation-unit error readers (defined in each .cu)
int csa2_read_and_clear_codec_error(cudaStream_t s);
int csa2_read_and_clear_index_error(cudaStream_t s);
int csa2_read_and_clear_topk_error(cudaStream_t s);
int csa2_read_and_clear_attn_error(cudaStream_t s);
