// cta_select.cuh -- exact Top-K of a small candidate set in shared memory,
// for a group of warps inside a larger CTA (the decode scan's epilogue).
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", section
// 2.3: the indexer keeps the Top-K entries of every query. Order: larger
// score key first, then smaller position (the same order as the Top-K
// kernels). Candidates are (key, position) pairs, key = score_key(score).
#pragma once

#include "common.cuh"

namespace csa2 {
namespace ctasel {

constexpr int kDigitBits = 8;
constexpr int kBins = 1 << kDigitBits;

// The group of warps that runs the selection: `nthreads` threads starting at
// thread 0 of the CTA, meeting at named barrier `bar_id`.
struct Group {
  int bar_id;
  int nthreads;
  __device__ __forceinline__ void sync() const {
    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(nthreads) : "memory");
  }
};

// AND of `pred` over the group's threads; also a barrier of the group.
__device__ __forceinline__ bool group_all(const Group& g, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(g.bar_id), "r"(g.nthreads)
      : "memory");
  return r != 0;
}

// The value a pass orders by: the key, or (ties pass) the complement of the
// position for entries whose key equals `tie` and 0 for the others, so that
// the largest values are the smallest positions of the ties.
__device__ __forceinline__ uint32_t sel_value(uint2 e, bool ties, uint32_t tie) {
  return ties ? (e.x == tie ? ~e.y : 0u) : e.x;
}

// need-th largest value (1-based) among c[0..n): returns it and, in *above,
// how many values are strictly larger. Needs need <= n (ties pass: need <=
// the number of ties). hist: kBins words; scr: 40 words. All threads of the
// group call it.
__device__ uint32_t select_value(const uint2* c, int n, uint32_t need, bool ties, uint32_t tie, const Group& g,
                                 uint32_t* hist, uint32_t* scr, uint32_t* above) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0, gone = 0;   // value bits fixed so far; count of values above the prefix
  for (int shift = 32 - kDigitBits; shift >= 0; shift -= kDigitBits) {
    const uint32_t mask_hi = shift + kDigitBits >= 32 ? 0u : ~0u << (shift + kDigitBits);
    for (int i = tid; i < kBins; i += g.nthreads) hist[i] = 0u;
    g.sync();
    for (int i = tid; i < n; i += g.nthreads) {
      const uint32_t v = sel_value(c[i], ties, tie);
      if ((v & mask_hi) == prefix) atomicAdd(&hist[(v >> shift) & (kBins - 1)], 1u);
    }
    g.sync();
    // running count from the top bin: thread t owns the kBins / nthreads bins
    // below kBins - t * (kBins / nthreads)
    const int per = kBins / g.nthreads;
    uint32_t local = 0;
    for (int j = 0; j < per; ++j) local += hist[kBins - 1 - tid * per - j];
    uint32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    if (lane == 31) scr[warp] = incl;
    g.sync();
    uint32_t wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += scr[w];
    const uint32_t excl = wbase + incl - local;
    const uint32_t want = need - gone;   // still needed inside this prefix
    if (excl < want && excl + local >= want) {
      uint32_t run = excl;
      for (int j = 0; j < per; ++j) {
        const int bin = kBins - 1 - tid * per - j;
        const uint32_t h = hist[bin];
        if (run + h >= want) {
          scr[32] = (uint32_t)bin;
          scr[33] = run;
          break;
        }
        run += h;
      }
    }
    g.sync();
    prefix |= scr[32] << shift;
    gone += scr[33];
    g.sync();
  }
  *above = gone;
  return prefix;
}

// Keeps, in place, the top `k` of c[0..n) by (key desc, position asc) and
// returns how many are kept (min(k, n)); *kth_key receives the key of the
// k-th (0 when n <= k: every key stays eligible).
__device__ int select_topk_inplace(uint2* c, int n, int k, const Group& g, uint32_t* hist, uint32_t* scr,
                                   uint32_t* kth_key) {
  if (n <= k) {
    *kth_key = 0u;
    return n;
  }
  uint32_t above;
  const uint32_t T = select_value(c, n, (uint32_t)k, false, 0u, g, hist, scr, &above);
  const uint32_t quota = (uint32_t)k - above;   // ties at T to keep (>= 1)
  // ties at T: keep the `quota` smallest positions (largest ~position)
  uint32_t ties = 0;
  {
    const int tid = threadIdx.x;
    uint32_t t = 0;
    for (int i = tid; i < n; i += g.nthreads) t += c[i].x == T;
    for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if ((tid & 31) == 0) scr[tid >> 5] = t;
    g.sync();
    for (int w = 0; w < (g.nthreads >> 5); ++w) ties += scr[w];
    g.sync();
  }
  uint32_t pos_cut = 0u;   // complement of the largest position kept among the ties
  bool cut = ties > quota;
  if (cut) {
    uint32_t a2;
    pos_cut = select_value(c, n, quota, true, T, g, hist, scr, &a2);
  }
  // compaction: thread t keeps a contiguous run of entries (order inside the
  // buffer carries no meaning), then a group scan places them
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + g.nthreads - 1) / g.nthreads;
  const int lo = tid * per, hi = min(n, lo + per);
  constexpr int kMaxPer = 16;   // n <= 16 x the group's threads
  uint2 e[kMaxPer];
  uint32_t kp = 0;              // bit j: entry lo + j is kept
#pragma unroll
  for (int j = 0; j < kMaxPer; ++j) {
    const int i = lo + j;
    e[j] = i < hi ? c[i] : make_uint2(0u, 0u);
    const bool keep = i < hi && (e[j].x > T || (e[j].x == T && (!cut || ~e[j].y >= pos_cut)));
    kp |= (uint32_t)keep << j;
  }
  const int nk = __popc(kp);
  uint32_t incl = (uint32_t)nk;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) scr[warp] = incl;
  g.sync();
  uint32_t base = 0, total = 0;
  for (int w = 0; w < (g.nthreads >> 5); ++w) {
    if (w < warp) base += scr[w];
    total += scr[w];
  }
  base += incl - (uint32_t)nk;
  g.sync();   // every thread has read its run before any is overwritten
  uint32_t r = base;
#pragma unroll
  for (int j = 0; j < kMaxPer; ++j)
    if (kp & (1u << j)) {
      if (r < (uint32_t)k) c[r] = e[j];
      ++r;
    }
  g.sync();
  *kth_key = T;
  return (int)min(total, (uint32_t)k);
}

}  // namespace ctasel
}  // namespace csa2
