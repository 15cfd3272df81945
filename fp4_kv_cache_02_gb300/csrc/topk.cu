// topk.cu -- Top-K selection and the hierarchical block pool.
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", section
// 2.3 (the indexer selects the Top-K entries for each query) and section 2.3.2
// with Figure 5 (each block of positions takes the maximum index score among
// its positions; the highest-scoring blocks form the candidate pool).
//
// Radix/threshold select on order-preserving 32-bit keys of the fp32 scores:
//   1. histogram of the top 11 key bits per row (shared-memory histogram per
//      CTA, flushed to a per-row global histogram; the decode scan builds it
//      in its epilogue);
//   2. select: the row is cut into regions of 4096 scores (more for very long
//      rows), one CTA each. While the region's loads are in flight the CTA
//      finds the threshold bin t of the row (the bin in which the running
//      count from the top reaches k). Every key in bin t or above is written,
//      in position order, to the region's own slice of the candidate buffer
//      (no global atomics), and the keys inside bin t are counted in a
//      second-level histogram of the next 11 key bits;
//   3. finalize, one CTA per row: the second-level threshold bin t2 splits the
//      candidates into taken ones and the few inside t2, which are ranked
//      exactly (key, then smaller position). The taken keys are compacted in
//      list order, which is ascending position when the row is dense, so the
//      ascending output needs no sort: the few exact-rank winners are merged
//      in by binary search. Rows given through a positions map are sorted at
//      the end unless already ascending.
// Indexer scores crowd into a narrow band of values, so one 11-bit level
// leaves thousands of candidates in bin t at a million entries; the second
// level cuts that to a handful. The result does not depend on the order in
// which CTAs run.
#include "common.cuh"

#include <mutex>

namespace csa2 {

__device__ int g_topk_error = 0;

constexpr int kHistBits = kTopkHistBits;  // 12: first level, top key bits
constexpr int kHistBins = kTopkHistBins;  // 4096
constexpr int kHist2Bits = 11;            // second level, the next key bits of bin t
constexpr int kHist2Bins = 1 << kHist2Bits;
constexpr int kRadixBits = 11;            // bits per pass of the exact radix select
constexpr int kRadixBins = 1 << kRadixBits;
constexpr int kSelThreads = 256;
constexpr int kPerThread = 16;                      // consecutive scores per select thread
constexpr int kSelTile = kSelThreads * kPerThread;  // 4096 scores
constexpr int kMaxRegions = 8192;                   // regions per row (their offsets live in shared memory)
constexpr int kFinThreads = 512;
constexpr int kFinPerThread = 4;
constexpr int kTieCap = 1024;                       // second-level ties ranked in shared memory
constexpr int kHist2Shift = 32 - kHistBits - kHist2Bits;  // 9: second-level digit is key bits [19, 9]

struct RowCounters {
  int32_t t;       // threshold bin (-1: fewer candidates than k)
  uint32_t above;  // candidates in bins above t
  uint32_t pad[5];
  int32_t scan_tiles;  // tiles claimed by the decode scan that fills the histogram
};
static_assert(sizeof(RowCounters) == 32 && offsetof(RowCounters, scan_tiles) % 4 == 0, "row counter layout");

struct TopkWs {
  uint32_t* hist;     // [B][kHistBins]  top 12 key bits
  uint32_t* hist2;    // [B][kHist2Bins] next 11 key bits of the keys in bin t
  RowCounters* cnt;   // [B]
  uint32_t* rcount;   // [B][n_regions]  keys each region wrote
  uint2* cand;        // [B][n]  (key, position); region r owns [r*region, r*region + its scores)
  int64_t region;     // scores per region (a multiple of kSelTile)
  int32_t n_regions;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Regions of m tiles of kSelTile scores. m = 1 (the most parallel select) until
// the launch holds more than kSelTilesPerLaunch tiles (rows x tiles a row):
// then each CTA walks up to 8 tiles, so that the per-CTA work (the row's
// histogram read, the threshold search, the second-level flush) is paid once
// per several tiles (4,096 prefill rows of 131,072 scores: 4 regions a row).
constexpr int64_t kSelTilesPerLaunch = 8192;
__host__ __device__ inline void topk_regions(int32_t B, int64_t n, int64_t* region, int32_t* n_regions) {
  const int64_t tiles = n > 0 ? (n + kSelTile - 1) / kSelTile : 1;
  int64_t m = (tiles + kMaxRegions - 1) / kMaxRegions;
  const int64_t all = (int64_t)(B > 0 ? B : 1) * tiles;
  if (all > kSelTilesPerLaunch) {
    int64_t mt = (all + kSelTilesPerLaunch - 1) / kSelTilesPerLaunch;
    mt = mt > 8 ? 8 : mt;
    mt = mt > tiles ? tiles : mt;
    m = m > mt ? m : mt;
  }
  *region = m * kSelTile;
  *n_regions = (int32_t)((tiles + m - 1) / m);
}

__host__ __device__ inline size_t topk_ws_layout(int32_t B, int64_t n, int32_t k, TopkWs* ws, char* base) {
  (void)k;
  int64_t region;
  int32_t nr;
  topk_regions(B, n, &region, &nr);
  size_t off = 0;
  size_t hist = off;   off = align_up(off + (size_t)B * kHistBins * 4, 256);
  size_t hist2 = off;  off = align_up(off + (size_t)B * kHist2Bins * 4, 256);
  size_t cnt = off;    off = align_up(off + (size_t)B * sizeof(RowCounters), 256);
  size_t rcount = off; off = align_up(off + (size_t)B * nr * 4, 256);
  size_t cand = off;   off = align_up(off + (size_t)B * (size_t)(n > 0 ? n : 1) * 8, 256);
  if (ws) {
    ws->hist = (uint32_t*)(base + hist);
    ws->hist2 = (uint32_t*)(base + hist2);
    ws->cnt = (RowCounters*)(base + cnt);
    ws->rcount = (uint32_t*)(base + rcount);
    ws->cand = (uint2*)(base + cand);
    ws->region = region;
    ws->n_regions = nr;
  }
  return off;
}

// The histograms and counters (the leading part of the layout) start at zero.
__host__ __device__ inline size_t topk_ws_zero_bytes(int32_t B) {
  return align_up(align_up((size_t)B * kHistBins * 4, 256) + align_up((size_t)B * kHist2Bins * 4, 256) +
                      (size_t)B * sizeof(RowCounters),
                  256);
}

__device__ int find_threshold_bin(const uint32_t* h, int nbins, uint32_t need, uint32_t* above_out,
                                  uint32_t* scratch);

// ---- pass 1: histogram of the top kHistBits key bits --------------------------
__global__ void __launch_bounds__(kSelThreads) topk_hist_kernel(
    const float* __restrict__ scores, int64_t n, const int32_t* __restrict__ n_valid,
    const int32_t* __restrict__ positions, int64_t chunk, int32_t k, TopkWs ws) {
  pdl_begin();
  __shared__ uint32_t sh[kHistBins];
  const int b = blockIdx.y;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  const int64_t row_off = (int64_t)b * n;
  int64_t nv = n_valid ? min((int64_t)n_valid[b], n) : n;
  int64_t lo = (int64_t)blockIdx.x * chunk, hi = min(lo + chunk, nv);
  const bool has_pos = positions != nullptr;
  for (int64_t sub = lo; sub < hi; sub += (int64_t)kSelThreads * 16) {
    // all loads of the sub-chunk in flight first: predicated, nothing reads
    // them before the last one is issued
    float sv[16];
    int32_t pv[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int64_t i = sub + (int64_t)e * kSelThreads + threadIdx.x;
      const bool in = i < hi;
      sv[e] = in ? scores[row_off + i] : __uint_as_float(0x7fc00000u);
      pv[e] = in && has_pos ? positions[row_off + i] : 0;
    }
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if (pv[e] >= 0 && score_is_candidate(sv[e])) atomicAdd(&sh[score_key(sv[e]) >> (32 - kHistBits)], 1u);
  }
  __syncthreads();
  uint32_t* gh = ws.hist + (size_t)b * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x)
    if (sh[i]) atomicAdd(&gh[i], sh[i]);
}

// Block-wide search, from the top bin down, for the first bin at which the
// running count reaches `need`. Returns the bin (-1 if the total is below
// `need`) and the count strictly above it. `h` has `nbins` entries in shared
// memory; nbins and blockDim.x are powers of two, nbins >= blockDim.x >= 32;
// `scratch` holds blockDim.x + 2 words. Thread j owns bins
// [nbins-(j+1)*per, nbins-j*per); a warp-shuffle scan over the threads finds
// the owner of the crossing.
__device__ int find_threshold_bin(const uint32_t* h, int nbins, uint32_t need, uint32_t* above_out,
                                  uint32_t* scratch) {
  const int per = nbins / blockDim.x;
  const int j = threadIdx.x, lane = j & 31, warp = j >> 5, nwarps = blockDim.x >> 5;
  const int top = nbins - j * per;
  uint32_t local = 0;
  for (int i = 0; i < per; ++i) local += h[top - 1 - ((i + j) & (per - 1))];  // rotated: no bank conflicts
  uint32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t wt = lane < nwarps ? scratch[lane] : 0u, wi = wt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += v;
    }
    __syncwarp();
    if (lane < nwarps) scratch[lane] = wi - wt;  // exclusive prefix of warp totals
  }
  __syncthreads();
  const uint32_t excl = scratch[warp] + incl - local;
  __syncthreads();
  if (excl < need && excl + local >= need) {
    uint32_t run = excl;
    for (int i = 1; i <= per; ++i) {
      const uint32_t c = h[top - i];
      if (run + c >= need) {
        scratch[blockDim.x] = (uint32_t)(top - i);
        scratch[blockDim.x + 1] = run;
        break;
      }
      run += c;
    }
  } else if (j == (int)blockDim.x - 1 && excl + local < need) {
    scratch[blockDim.x] = 0xFFFFFFFFu;       // total below need
    scratch[blockDim.x + 1] = excl + local;  // = total
  }
  __syncthreads();
  const int bin = (int)scratch[blockDim.x];
  *above_out = scratch[blockDim.x + 1];
  __syncthreads();
  return bin;
}

// One warp finds, in a global histogram of kHist2Bins counts, the first bin
// from the top at which the running count reaches `need` (-1 if the total is
// below it) and the count strictly above that bin. Lane l owns bins
// [kHist2Bins - 64(l+1), kHist2Bins - 64 l); a warp scan over the lanes finds the
// owning lane, then the lanes split that lane's 64 bins two apiece. The row
// must be 256-byte aligned; counts are read through L2 (__ldcg) because other
// CTAs of an earlier kernel wrote them with atomics.
// Sum of the 64 bins lane l owns (the loads can be issued before `need` is known).
__device__ __forceinline__ uint32_t warp_hist_lane_sum(const uint32_t* __restrict__ gh) {
  const int lane = threadIdx.x & 31;
  const uint4* p = reinterpret_cast<const uint4*>(gh + kHist2Bins - 64 * (lane + 1));
  uint4 v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __ldcg(p + i);
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) s += v[i].x + v[i].y + v[i].z + v[i].w;
  return s;
}

__device__ int warp_threshold_bin(const uint32_t* __restrict__ gh, uint32_t need, uint32_t* above_out,
                                  uint32_t* count_out = nullptr, const uint32_t* lane_sum = nullptr) {
  static_assert(kHist2Bins == 32 * 64, "one warp covers the histogram 64 bins a lane");
  const int lane = threadIdx.x & 31;
  const uint32_t s = lane_sum ? *lane_sum : warp_hist_lane_sum(gh);
  uint32_t incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
  if (total < need) {
    *above_out = total;
    return -1;
  }
  const int c = __ffs(__ballot_sync(0xffffffffu, incl >= need)) - 1;
  const uint32_t excl_c = __shfl_sync(0xffffffffu, incl - s, c);
  const int top_c = kHist2Bins - 64 * c;
  // lane l: bins top_c-1-2l (.y) and top_c-2-2l (.x)
  const uint2 v = __ldcg(reinterpret_cast<const uint2*>(gh + top_c - 2 - 2 * lane));
  const uint32_t ps = v.x + v.y;
  uint32_t incl2 = ps;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, incl2, o);
    if (lane >= o) incl2 += x;
  }
  const int c2 = __ffs(__ballot_sync(0xffffffffu, excl_c + incl2 >= need)) - 1;
  uint32_t base = excl_c + __shfl_sync(0xffffffffu, incl2 - ps, c2);
  const uint32_t hy = __shfl_sync(0xffffffffu, v.y, c2);
  const uint32_t hx = __shfl_sync(0xffffffffu, v.x, c2);
  int bin;
  if (base + hy >= need) {
    bin = top_c - 1 - 2 * c2;
    if (count_out) *count_out = hy;
  } else {
    bin = top_c - 2 - 2 * c2;
    base += hy;
    if (count_out) *count_out = hx;
  }
  *above_out = base;
  return bin;
}

// Exact r-th largest among `count` 32-bit keys (in global memory, key field of
// uint2 or the `x` values of an int array transform), restricted to those whose
// top `fixed_bits` equal `prefix`. Radix passes over the remaining bits with
// `bits_per_pass` bits each. Returns the full threshold key; *r_left is how
// many keys equal to the threshold are still needed.
template <typename KeyFn>
__device__ uint32_t radix_select_desc(int count, uint32_t need, int fixed_bits, uint32_t prefix,
                                      KeyFn keyfn, uint32_t* hist /*kRadixBins*/, uint32_t* scratch,
                                      uint32_t* r_left) {
  int done_bits = fixed_bits;
  while (done_bits < 32) {
    int pass_bits = min(kRadixBits, 32 - done_bits);
    int nb = 1 << pass_bits;
    int nbins = nb < (int)blockDim.x ? (int)blockDim.x : nb;  // pad to a multiple of blockDim
    for (int i = threadIdx.x; i < nbins; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    int shift = 32 - done_bits - pass_bits;
    for (int i = threadIdx.x; i < count; i += blockDim.x) {
      uint32_t key = keyfn(i);
      bool match = done_bits == 0 ? true : ((key >> (32 - done_bits)) == (prefix >> (32 - done_bits)));
      if (match) atomicAdd(&hist[(key >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    uint32_t above;
    int bin = find_threshold_bin(hist, nbins, need, &above, scratch);
    // bin >= 0 always: callers guarantee at least `need` matching keys
    prefix |= ((uint32_t)bin) << shift;
    need -= above;
    done_bits += pass_bits;
  }
  *r_left = need;
  return prefix;
}

// Ascending bitonic sort of a[0..n2) in shared memory, n2 = E * blockDim.x
// (blockDim.x a multiple of 32, E a power of two <= 16). Thread (warp w, lane
// l) keeps the E elements w*32E + r*32 + l in registers: partners less than 32
// apart are exchanged with shuffles, those within a warp's run in registers,
// and only strides of 32E and more go through shared memory.
template <int E>
__device__ void block_sort_asc_e(int32_t* a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n2 = E * (int)blockDim.x;
  const int base = warp * 32 * E + lane;
  int32_t v[E];
#pragma unroll
  for (int r = 0; r < E; ++r) v[r] = a[base + r * 32];
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 32 * E) {
        __syncthreads();
#pragma unroll
        for (int r = 0; r < E; ++r) a[base + r * 32] = v[r];
        __syncthreads();
#pragma unroll
        for (int r = 0; r < E; ++r) {
          const int e = base + r * 32;
          const int32_t y = a[e ^ stride];
          const bool keep_min = ((e & stride) == 0) == ((e & size) == 0);
          v[r] = keep_min ? min(v[r], y) : max(v[r], y);
        }
      } else if (stride >= 32) {
        // partners are registers r and r ^ (stride / 32); unrolled over the
        // possible strides so every register index is a compile-time constant
#pragma unroll
        for (int rs = 1; rs < E; rs <<= 1) {
          if (rs == (stride >> 5)) {
            int32_t w[E];
#pragma unroll
            for (int r = 0; r < E; ++r) {
              const int e = base + r * 32;
              const bool keep_min = ((r & rs) == 0) == ((e & size) == 0);
              w[r] = keep_min ? min(v[r], v[r ^ rs]) : max(v[r], v[r ^ rs]);
            }
#pragma unroll
            for (int r = 0; r < E; ++r) v[r] = w[r];
          }
        }
      } else {
#pragma unroll
        for (int r = 0; r < E; ++r) {
          const int e = base + r * 32;
          const int32_t y = __shfl_xor_sync(0xffffffffu, v[r], stride);
          const bool keep_min = ((lane & stride) == 0) == ((e & size) == 0);
          v[r] = keep_min ? min(v[r], y) : max(v[r], y);
        }
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < E; ++r) a[base + r * 32] = v[r];
  __syncthreads();
}

// n2 a power of two, blockDim.x <= n2 <= 16 * blockDim.x.
__device__ void block_sort_asc(int32_t* a, int n2) {
  switch (n2 / (int)blockDim.x) {
    case 1: block_sort_asc_e<1>(a); break;
    case 2: block_sort_asc_e<2>(a); break;
    case 4: block_sort_asc_e<4>(a); break;
    case 8: block_sort_asc_e<8>(a); break;
    default: block_sort_asc_e<16>(a); break;
  }
}

// Exclusive prefix sum of v over the block (blockDim.x a multiple of 32,
// <= 1024); *total receives the block sum. `sh` holds 33 words.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* total, uint32_t* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t wt = lane < nwarps ? sh[lane] : 0u;
    uint32_t wi = wt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += x;
    }
    if (lane < nwarps) sh[lane] = wi - wt;
    if (lane == 31) sh[32] = wi;
  }
  __syncthreads();
  const uint32_t r = sh[warp] + incl - v;
  *total = sh[32];
  __syncthreads();
  return r;
}

// Block-wide exclusive scan with one barrier: each warp publishes its total in
// `buf` (one word per warp), and every thread sums the totals of the warps
// before its own. Consecutive calls must alternate between two buffers: a
// buffer is written again only after every thread has passed the barrier of
// the call in between, so after it has been read.
__device__ __forceinline__ uint32_t block_exclusive_scan_1bar(uint32_t v, uint32_t* total, uint32_t* buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) buf[warp] = incl;
  __syncthreads();
  uint32_t before = 0, tot = 0;
  for (int w = 0; w < nwarps; ++w) {
    const uint32_t x = buf[w];
    before += w < warp ? x : 0u;
    tot += x;
  }
  *total = tot;
  return before + incl - v;
}

// ---- pass 2: every key in bin t or above, written per region in order ------
// Loads the kPerThread consecutive scores [i0, i0 + kPerThread) of a row (16-byte
// vectors when the row allows) and returns the mask of candidates.
template <bool kPositions>
__device__ __forceinline__ uint32_t load_run(const float* __restrict__ scores, const int32_t* __restrict__ positions,
                                             int64_t row_off, int64_t i0, int64_t nv, bool vec, uint32_t* key,
                                             int32_t* pos) {
  float s[kPerThread];
  int32_t p[kPerThread];
  if (vec && i0 + kPerThread <= nv) {
    const float4* sp = reinterpret_cast<const float4*>(scores + row_off + i0);
#pragma unroll
    for (int q = 0; q < kPerThread / 4; ++q) {
      const float4 v = sp[q];
      s[4 * q] = v.x; s[4 * q + 1] = v.y; s[4 * q + 2] = v.z; s[4 * q + 3] = v.w;
    }
    if (kPositions) {
      const int4* pp = reinterpret_cast<const int4*>(positions + row_off + i0);
#pragma unroll
      for (int q = 0; q < kPerThread / 4; ++q) {
        const int4 v = pp[q];
        p[4 * q] = v.x; p[4 * q + 1] = v.y; p[4 * q + 2] = v.z; p[4 * q + 3] = v.w;
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const bool in = i0 + e < nv;
      s[e] = in ? scores[row_off + i0 + e] : __uint_as_float(0x7fc00000u);
      if (kPositions) p[e] = in ? positions[row_off + i0 + e] : -1;
    }
  }
  uint32_t ok = 0;
#pragma unroll
  for (int e = 0; e < kPerThread; ++e) {
    const int32_t pe = kPositions ? p[e] : (int32_t)(i0 + e);
    ok |= (uint32_t)(i0 + e < nv && pe >= 0 && score_is_candidate(s[e])) << e;
    key[e] = score_key(s[e]);
    if (kPositions) pos[e] = pe;
  }
  return ok;
}

template <bool kPositions>
__global__ void __launch_bounds__(kSelThreads, 4) topk_select_kernel(
    const float* __restrict__ scores, int64_t n, const int32_t* __restrict__ n_valid,
    const int32_t* __restrict__ positions, int32_t k, TopkWs ws) {
  pdl_begin();
  __shared__ uint32_t h2[kHist2Bins];
  __shared__ uint32_t s_wsum[kSelThreads / 32];
  __shared__ uint32_t s_wex[kSelThreads / 32];
  __shared__ uint32_t s_scan[33];
  __shared__ int s_t;
  const int b = blockIdx.y;
  const int r = blockIdx.x;
  const int64_t row_off = (int64_t)b * n;
  const int64_t nv = n_valid ? min((int64_t)n_valid[b], n) : n;
  const int64_t lo_r = (int64_t)r * ws.region;
  uint32_t* rcount = ws.rcount + (size_t)b * ws.n_regions;
  if (lo_r >= nv && r != 0) {  // region 0 always runs: it records t
    if (threadIdx.x == 0) rcount[r] = 0u;
    return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool vec = (((uintptr_t)(scores + row_off)) & 15) == 0 &&
                   (!kPositions || (((uintptr_t)(positions + row_off)) & 15) == 0);
  // this thread's loads go out first; the threshold search overlaps them
  uint32_t key[kPerThread];
  int32_t pos[kPositions ? kPerThread : 1];
  int64_t lo = lo_r;
  uint32_t ok = lo < nv ? load_run<kPositions>(scores, positions, row_off, lo + (int64_t)threadIdx.x * kPerThread,
                                               nv, vec, key, pos)
                        : 0u;
  // threshold bin t of the row: thread j sums the 16 bins [4080 - 16j, 4096 - 16j),
  // a block scan from the top finds the thread whose bins reach k
  constexpr int kBinsPerThread = kHistBins / kSelThreads;
  static_assert(kBinsPerThread == 16, "16 histogram bins per select thread");
  const uint4* hp = reinterpret_cast<const uint4*>(ws.hist + (size_t)b * kHistBins +
                                                   kHistBins - kBinsPerThread * (threadIdx.x + 1));
  uint4 hv[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) hv[q] = __ldcg(hp + q);  // bins base + 4q .. base + 4q + 3
  for (int i = threadIdx.x; i < kHist2Bins; i += kSelThreads) h2[i] = 0u;
  uint32_t hs = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) hs += hv[q].x + hv[q].y + hv[q].z + hv[q].w;
  uint32_t hin = hs;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, hin, o);
    if (lane >= o) hin += x;
  }
  if (lane == 31) s_wsum[warp] = hin;
  __syncthreads();
  if (warp == 0) {
    constexpr int kWarps = kSelThreads / 32;
    const uint32_t wv = lane < kWarps ? s_wsum[lane] : 0u;
    uint32_t wi = wv;
#pragma unroll
    for (int o = 1; o < kWarps; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += x;
    }
    if (lane < kWarps) s_wex[lane] = wi - wv;
    if (lane == kWarps - 1 && wi < (uint32_t)k) {  // fewer candidates than k
      s_t = -1;
      if (r == 0) {
        ws.cnt[b].t = -1;
        ws.cnt[b].above = wi;
      }
    }
  }
  __syncthreads();
  {
    const uint32_t hex = s_wex[warp] + hin - hs;  // count in the bins above this thread's
    if (hex < (uint32_t)k && hex + hs >= (uint32_t)k) {
      uint32_t v[kBinsPerThread];  // top bin first
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[15 - 4 * q] = hv[q].x;
        v[14 - 4 * q] = hv[q].y;
        v[13 - 4 * q] = hv[q].z;
        v[12 - 4 * q] = hv[q].w;
      }
      uint32_t run = hex, cnt_t = v[kBinsPerThread - 1];
      int bin = kHistBins - kBinsPerThread * (int)threadIdx.x - 1;
#pragma unroll
      for (int i = 0; i < kBinsPerThread - 1; ++i) {
        if (run + v[i] >= (uint32_t)k) {
          cnt_t = v[i];
          break;
        }
        run += v[i];
        --bin;
      }
      s_t = bin;
      if (r == 0) {
        ws.cnt[b].t = bin;
        ws.cnt[b].above = run;
        ws.cnt[b].pad[0] = cnt_t;  // keys in bin t
      }
    }
  }
  __syncthreads();
  const int t = s_t;
  const int64_t hi_r = min(lo_r + ws.region, nv);
  uint2* cand = ws.cand + row_off;
  uint32_t written = 0;  // keys this region wrote so far (same in every thread)
  bool any_t = false;
  for (;;) {
    uint32_t flag = 0;
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int digit = (int)(key[e] >> (32 - kHistBits));
      const bool f = ((ok >> e) & 1u) && digit >= t;
      flag |= (uint32_t)f << e;
      if (f && digit == t) {
        atomicAdd(&h2[(key[e] >> kHist2Shift) & (kHist2Bins - 1)], 1u);
        any_t = true;
      }
    }
    uint32_t total;
    const uint32_t excl = block_exclusive_scan((uint32_t)__popc(flag), &total, s_scan);
    if (flag) {
      int64_t o = lo_r + written + excl;
#pragma unroll
      for (int e = 0; e < kPerThread; ++e) {
        if ((flag >> e) & 1u) {
          const int32_t p = kPositions ? pos[kPositions ? e : 0] : (int32_t)(lo + (int64_t)threadIdx.x * kPerThread + e);
          if (o < hi_r) cand[o] = make_uint2(key[e], (uint32_t)p);
          else record_error(&g_topk_error, CSA2_ERR_DEVICE);
          ++o;
        }
      }
    }
    written += total;
    lo += kSelTile;
    if (lo >= hi_r) break;
    ok = load_run<kPositions>(scores, positions, row_off, lo + (int64_t)threadIdx.x * kPerThread, nv, vec, key, pos);
  }
  if (threadIdx.x == 0) rcount[r] = written;
  if (__syncthreads_or(any_t)) {
    uint32_t* gh2 = ws.hist2 + (size_t)b * kHist2Bins;
    for (int i = threadIdx.x; i < kHist2Bins; i += kSelThreads)
      if (h2[i]) atomicAdd(&gh2[i], h2[i]);
  }
}

// ---- passes 1 + 2 in one, for batches of many long dense rows -------------
// One CTA per row reads the row once, a tile of kSelTile scores at a time (the
// next tile's loads in flight while the current one is processed). Each tile
// goes into the shared-memory histogram, and its keys at or above the running
// threshold bin are appended, in position order, to their region's slice. The
// running bin is the threshold bin of the histogram so far, recomputed after
// each of the first four tiles and then after every eighth: it only rises as
// keys arrive and never passes the row's final threshold bin t, so the slices
// hold every key of bin t and above (and some below it). At the end the exact
// t is found, each slice is compacted in place to its keys in bin t or above,
// and the keys in bin t are counted in the second-level histogram: the
// workspace then holds what the histogram and select kernels leave for the
// finalize. Scores move as raw 32-bit words and are keyed with integer
// operations only, so no NaN passes through a float register.
constexpr uint32_t kCandKeyLo = 0x00800000u;  // score_key(-inf) + 1
constexpr uint32_t kCandKeyHi = 0xff800000u;  // score_key(+inf)
constexpr uint32_t kNotCandidateBits = 0xffffffffu;  // a negative NaN: key 0
// score_key() of the fp32 score whose bit pattern is b, in integer operations
__device__ __forceinline__ uint32_t key_of_bits(uint32_t b) {
  return b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u);
}

__global__ void __launch_bounds__(kSelThreads, 4) topk_collect_kernel(const float* __restrict__ scores, int64_t n,
                                                                      const int32_t* __restrict__ n_valid, int32_t k,
                                                                      TopkWs ws) {
  pdl_begin();
  __shared__ uint32_t sh[kHistBins];
  __shared__ uint32_t h2[kHist2Bins];
  __shared__ uint32_t scratch[kSelThreads + 2];
  __shared__ uint32_t s_wsum[2][kSelThreads / 32];  // the tile loop's scans, alternating
  __shared__ uint32_t s_scan[33];
  const int b = blockIdx.x;
  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) sh[i] = 0u;
  for (int i = threadIdx.x; i < kHist2Bins; i += kSelThreads) h2[i] = 0u;
  __syncthreads();
  const int64_t row_off = (int64_t)b * n;
  const int64_t nv = n_valid ? max((int64_t)0, min((int64_t)n_valid[b], n)) : n;
  const uint32_t* wrow = reinterpret_cast<const uint32_t*>(scores + row_off);
  const bool vec = (((uintptr_t)wrow) & 15) == 0;
  uint2* cand = ws.cand + row_off;
  uint32_t* rcount = ws.rcount + (size_t)b * ws.n_regions;
  int t_run = -1;        // threshold bin of the histogram so far (-1: fewer than k keys)
  uint32_t written = 0;  // superset entries of the current region
  int reg = 0;           // current region
  uint32_t nx[kPerThread];
  auto load_tile = [&](int64_t i0) {
    if (vec && i0 + kPerThread <= nv) {
      const uint4* sp = reinterpret_cast<const uint4*>(wrow + i0);
#pragma unroll
      for (int q = 0; q < kPerThread / 4; ++q) {
        const uint4 v = __ldcs(sp + q);
        nx[4 * q] = v.x; nx[4 * q + 1] = v.y; nx[4 * q + 2] = v.z; nx[4 * q + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < kPerThread; ++e) nx[e] = i0 + e < nv ? wrow[i0 + e] : kNotCandidateBits;
    }
  };
  if (nv > 0) load_tile((int64_t)threadIdx.x * kPerThread);
  int j = 0;
  int64_t reg_lo = 0;    // first score of the current region (regions are whole tiles)
  for (int64_t lo = 0; lo < nv; lo += kSelTile, ++j) {
    if (lo >= reg_lo + ws.region) {  // the earlier region's superset is complete
      if (threadIdx.x == 0) rcount[reg] = written;
      ++reg;
      reg_lo += ws.region;
      written = 0;
    }
    uint32_t cur[kPerThread];
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) cur[e] = nx[e];
    const int64_t p0 = lo + (int64_t)threadIdx.x * kPerThread;
    if (lo + kSelTile < nv) load_tile(p0 + kSelTile);
    // a key is a candidate when it lies in [key(-inf) + 1, key(+inf)] (NaNs of
    // either sign, and the words loaded past n_valid, fall outside); it is
    // flagged when it is also at or above the running bin
    const uint32_t lo_flag = t_run > 0 ? max((uint32_t)t_run << (32 - kHistBits), kCandKeyLo) : kCandKeyLo;
    uint32_t flag = 0;
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const uint32_t key = key_of_bits(cur[e]);
      if (key - kCandKeyLo <= kCandKeyHi - kCandKeyLo) atomicAdd(&sh[key >> (32 - kHistBits)], 1u);
      flag |= (uint32_t)(key - lo_flag <= kCandKeyHi - lo_flag) << e;
    }
    uint32_t total;
    const uint32_t ex = block_exclusive_scan_1bar((uint32_t)__popc(flag), &total, s_wsum[j & 1]);
    if (flag) {
      int64_t o = reg_lo + written + ex;
#pragma unroll
      for (int e = 0; e < kPerThread; ++e)
        if ((flag >> e) & 1u) cand[o++] = make_uint2(key_of_bits(cur[e]), (uint32_t)(p0 + e));
    }
    written += total;
    if (j < 4 || (j & 7) == 7) {
      uint32_t above;
      t_run = find_threshold_bin(sh, kHistBins, (uint32_t)k, &above, scratch);  // (its barriers publish sh)
    }
  }
  if (threadIdx.x == 0) {
    rcount[reg] = written;
    for (int r = reg + 1; r < ws.n_regions; ++r) rcount[r] = 0u;  // past n_valid
  }
  // the exact threshold bin of the row and the counts the finalize reads
  // (the last tile's scan published the histogram)
  uint32_t above;
  const int t = find_threshold_bin(sh, kHistBins, (uint32_t)k, &above, scratch);
  if (threadIdx.x == 0) {
    ws.cnt[b].t = t;
    ws.cnt[b].above = above;
    ws.cnt[b].pad[0] = t >= 0 ? sh[t] : 0u;
  }
  // compaction of every region's slice to its keys in bin t or above, in
  // order, in place: a chunk is read into registers before the scan's barrier
  // and written after it, and the writes never pass the chunk's reads. The
  // slices and their counts were written by this CTA before a barrier, so they
  // are read with plain loads (an L2-only load may not see them yet).
  bool any_t = false;
  for (int r = 0; r <= reg; ++r) {
    const uint32_t m = rcount[r];
    uint2* sl = cand + (int64_t)r * ws.region;
    uint32_t kept = 0;
    for (uint32_t base = 0; base < m; base += (uint32_t)kSelThreads * 4) {
      uint2 c[4];
      uint32_t f = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t g = base + threadIdx.x * 4 + e;
        if (g < m) {
          c[e] = sl[g];
          const int digit = (int)(c[e].x >> (32 - kHistBits));
          f |= (uint32_t)(digit >= t) << e;
          if (digit == t) {
            atomicAdd(&h2[(c[e].x >> kHist2Shift) & (kHist2Bins - 1)], 1u);
            any_t = true;
          }
        }
      }
      uint32_t tot;
      const uint32_t ex = block_exclusive_scan((uint32_t)__popc(f), &tot, s_scan);
      uint32_t o = kept + ex;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if ((f >> e) & 1u) sl[o++] = c[e];
      kept += tot;
      __syncthreads();   // this chunk's writes land before the next chunk is read
    }
    if (threadIdx.x == 0) rcount[r] = kept;
  }
  if (__syncthreads_or(any_t)) {
    uint32_t* gh2 = ws.hist2 + (size_t)b * kHist2Bins;
    for (int i = threadIdx.x; i < kHist2Bins; i += kSelThreads)
      if (h2[i]) gh2[i] = h2[i];
  }
}

// Appends every entry [0, count) of `ld` to out (through the s_nout ticket).
template <typename LoadFn>
__device__ void take_all(uint32_t count, LoadFn ld, int32_t k, int32_t* out, uint32_t& s_nout) {
  for (uint32_t i = threadIdx.x; i < count; i += blockDim.x) {
    const uint32_t slot = atomicAdd(&s_nout, 1u);
    if (slot < (uint32_t)k) out[slot] = (int32_t)ld(i).y;
  }
}

// Takes the `need` largest of `count` (key, position) entries read through
// `ld`, every key's top `fixed_bits` equal to those of `prefix`: keys above the
// exact threshold key T are taken, and among keys equal to T the smallest
// positions. h has kRadixBins words (or blockDim.x if more), scratch
// blockDim.x + 8.
template <typename LoadFn>
__device__ void resolve_exact(uint32_t count, uint32_t need, int fixed_bits, uint32_t prefix, LoadFn ld, int32_t k,
                              int32_t* out, uint32_t& s_nout, uint32_t* h, uint32_t* scratch) {
  if (need >= count) {
    take_all(count, ld, k, out, s_nout);
    return;
  }
  uint32_t r2;
  const uint32_t T = radix_select_desc(
      (int)count, need, fixed_bits, prefix, [&](int i) { return ld((uint32_t)i).x; }, h, scratch, &r2);
  __shared__ uint32_t s_eq, s_r3;
  if (threadIdx.x == 0) {
    s_eq = 0;
    s_r3 = 0;
  }
  __syncthreads();
  uint32_t local = 0;
  for (uint32_t i = threadIdx.x; i < count; i += blockDim.x) local += (ld(i).x == T);
  atomicAdd(&s_eq, local);
  __syncthreads();
  const uint32_t n_eq = s_eq;
  const bool all_eq = r2 >= n_eq;
  uint32_t P = 0xFFFFFFFFu, r3 = 0;
  if (!all_eq) {
    // positions are >= 0, so ~position has bit 31 set: select the r2 largest
    // ~position among keys == T
    P = radix_select_desc(
        (int)count, r2, 0, 0u,
        [&](int i) {
          const uint2 c = ld((uint32_t)i);
          return c.x == T ? ~c.y : 0u;
        },
        h, scratch, &r3);
  }
  // keys above T, ties at T with ~position above P, and r3 of the ties sitting
  // exactly at ~position == P (a ticket: they share one position)
  for (uint32_t i = threadIdx.x; i < count; i += blockDim.x) {
    const uint2 c = ld(i);
    bool tk = c.x > T || (c.x == T && (all_eq || (~c.y) > P));
    if (!tk && !all_eq && c.x == T && ~c.y == P) tk = atomicAdd(&s_r3, 1u) < r3;
    if (tk) {
      const uint32_t slot = atomicAdd(&s_nout, 1u);
      if (slot < (uint32_t)k) out[slot] = (int32_t)c.y;
    }
  }
}

// Region holding flat list index g: the largest j in [0, R) with prefix[j] <= g.
__device__ __forceinline__ int region_of(const uint32_t* prefix, int R, uint32_t g) {
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= g) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Number of entries of the ascending array a[0..len) that are below v.
__device__ __forceinline__ uint32_t count_below(const int32_t* a, uint32_t len, int32_t v) {
  uint32_t lo = 0, hi = len;
  while (lo < hi) {
    const uint32_t mid = (lo + hi) >> 1;
    if (a[mid] < v) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// ---- pass 3: one CTA per row resolves bin t and writes the row -------------
// Shared memory (dynamic): ties (uint2) [kTieCap], prefix [kMaxRegions + 1],
// out [CSA2_MAX_TOPK], h [kRadixBins], scratch [kFinThreads + 8], tsel [kTieCap].
static constexpr size_t kFinSmem =
    (size_t)kTieCap * 8 + (size_t)(kMaxRegions + 1 + CSA2_MAX_TOPK + kRadixBins + kFinThreads + 8 + kTieCap) * 4;

__global__ void __launch_bounds__(kFinThreads, 1) topk_finalize_kernel(int64_t n, int32_t k, TopkWs ws,
                                                                       int32_t* __restrict__ idx, int dense) {
  pdl_begin();
  extern __shared__ __align__(16) unsigned char fsm[];
  uint2* ties = reinterpret_cast<uint2*>(fsm);
  uint32_t* prefix = reinterpret_cast<uint32_t*>(fsm + (size_t)kTieCap * 8);
  int32_t* out = reinterpret_cast<int32_t*>(prefix + kMaxRegions + 1);
  uint32_t* h = reinterpret_cast<uint32_t*>(out + CSA2_MAX_TOPK);
  uint32_t* scratch = h + kRadixBins;
  int32_t* tsel = reinterpret_cast<int32_t*>(scratch + kFinThreads + 8);
  __shared__ uint32_t s_nout, s_ntie, s_nsel, s_above2, s_ct2;
  __shared__ int s_t2;
  const int b = blockIdx.x;
  const int R = ws.n_regions;
  const int64_t row_off = (int64_t)b * n;
  const uint2* cand = ws.cand + row_off;
  int32_t* dst = idx + (size_t)b * k;
  // the row's counters, its region sizes and (warp 0) its second-level
  // histogram are loaded together
  uint32_t h2_sum = 0;
  if (threadIdx.x < 32) h2_sum = warp_hist_lane_sum(ws.hist2 + (size_t)b * kHist2Bins);
  const int t = __ldcg(&ws.cnt[b].t);
  const uint32_t above = __ldcg(&ws.cnt[b].above);
  const uint32_t c_t = t >= 0 ? __ldcg(&ws.cnt[b].pad[0]) : 0u;  // keys in bin t, recorded by the select
  const uint32_t r = t >= 0 ? (uint32_t)k - above : 0u;  // still needed from bin t
  const bool need_res = t >= 0 && r < c_t;
  // region sizes -> offsets (the loads are in flight while warp 0 finds t2)
  const uint32_t* rc = ws.rcount + (size_t)b * R;
  const int per = (R + kFinThreads - 1) / kFinThreads;
  const int j0 = (int)threadIdx.x * per, j1 = min(j0 + per, R);
  uint32_t local = 0;
  for (int j = j0; j < j1; ++j) local += __ldcg(rc + j);
  if (need_res && threadIdx.x < 32) {
    uint32_t above2, c2 = 0;
    const int t2 = warp_threshold_bin(ws.hist2 + (size_t)b * kHist2Bins, r, &above2, &c2, &h2_sum);
    if (threadIdx.x == 0) {
      s_t2 = t2;
      s_above2 = above2;
      s_ct2 = c2;
    }
  }
  if (threadIdx.x == 0) {
    s_nout = 0;
    s_ntie = 0;
    s_nsel = 0;
  }
  uint32_t total_m;
  uint32_t run = block_exclusive_scan(local, &total_m, scratch);
  for (int j = j0; j < j1; ++j) {
    prefix[j] = run;
    run += __ldcg(rc + j);
  }
  if (threadIdx.x == 0) prefix[R] = total_m;
  __syncthreads();
  const uint32_t M = total_m;
  int t2 = -1;
  uint32_t c_t2 = 0, r2 = 0;
  bool res_ties = false;
  if (need_res) {
    t2 = s_t2;
    if (t2 >= 0) {
      c_t2 = s_ct2;
      r2 = r - s_above2;
      res_ties = r2 < c_t2;
    }
  }
  const auto ld_flat = [&](uint32_t g) -> uint2 {
    const int j = region_of(prefix, R, g);
    return __ldcg(cand + (int64_t)j * ws.region + (g - prefix[j]));
  };
  bool sort_out = !dense;
  if (!need_res || (t2 >= 0 && c_t2 <= (uint32_t)kTieCap)) {
    // one ordered pass: keys above (t, t2) are compacted in list order; the
    // keys at (t, t2) are collected when only some of them are taken
    for (uint32_t base = 0; base < M; base += (uint32_t)kFinThreads * kFinPerThread) {
      const uint32_t g0 = base + threadIdx.x * kFinPerThread;
      uint2 c[kFinPerThread];
      uint32_t valid = 0;
      if (g0 < M) {
        int j = region_of(prefix, R, g0);
#pragma unroll
        for (int e = 0; e < kFinPerThread; ++e) {
          const uint32_t g = g0 + e;
          if (g < M) {
            while (j + 1 < R && prefix[j + 1] <= g) ++j;
            c[e] = __ldcg(cand + (int64_t)j * ws.region + (g - prefix[j]));
            valid |= 1u << e;
          }
        }
      }
      uint32_t def = 0;
#pragma unroll
      for (int e = 0; e < kFinPerThread; ++e) {
        if (!((valid >> e) & 1u)) continue;
        const int digit = (int)(c[e].x >> (32 - kHistBits));
        const int d2 = (int)((c[e].x >> kHist2Shift) & (kHist2Bins - 1));
        const bool at_t = need_res && digit == t;
        const bool taken = !at_t || d2 > t2 || (d2 == t2 && !res_ties);
        def |= (uint32_t)taken << e;
        if (at_t && d2 == t2 && res_ties) {
          const uint32_t slot = atomicAdd(&s_ntie, 1u);
          if (slot < (uint32_t)kTieCap) ties[slot] = c[e];
        }
      }
      uint32_t tot;
      const uint32_t ex = block_exclusive_scan((uint32_t)__popc(def), &tot, scratch);
      uint32_t o = s_nout + ex;
#pragma unroll
      for (int e = 0; e < kFinPerThread; ++e) {
        if ((def >> e) & 1u) {
          if (o < (uint32_t)k) out[o] = (int32_t)c[e].y;
          else record_error(&g_topk_error, CSA2_ERR_DEVICE);
          ++o;
        }
      }
      __syncthreads();
      if (threadIdx.x == 0) s_nout += tot;
      __syncthreads();
    }
    const uint32_t n_def = min(s_nout, (uint32_t)k);
    if (res_ties) {
      // exact rank of each tie: larger key first, then smaller position, then list slot
      const uint32_t nt = min(s_ntie, (uint32_t)kTieCap);
      for (uint32_t i = threadIdx.x; i < nt; i += kFinThreads) {
        const uint2 ci = ties[i];
        uint32_t rank = 0;
        for (uint32_t j = 0; j < nt; ++j) {
          const uint2 cj = ties[j];
          rank += (cj.x > ci.x) || (cj.x == ci.x && ((int32_t)cj.y < (int32_t)ci.y || (cj.y == ci.y && j < i)));
        }
        if (rank < r2) tsel[atomicAdd(&s_nsel, 1u)] = (int32_t)ci.y;
      }
      __syncthreads();
      const uint32_t nsel = s_nsel;
      if (dense) {
        // positions are distinct: sort the few winners by rank, then merge the
        // two ascending lists straight into the output row
        int32_t* tsorted = reinterpret_cast<int32_t*>(ties);
        for (uint32_t i = threadIdx.x; i < nsel; i += kFinThreads) {
          const int32_t v = tsel[i];
          uint32_t rank = 0;
          for (uint32_t j = 0; j < nsel; ++j) rank += tsel[j] < v;
          tsorted[rank] = v;
        }
        __syncthreads();
        for (uint32_t i = threadIdx.x; i < n_def; i += kFinThreads) {
          const int32_t q = out[i];
          const uint32_t d = i + count_below(tsorted, nsel, q);
          if (d < (uint32_t)k) dst[d] = q;
        }
        for (uint32_t j = threadIdx.x; j < nsel; j += kFinThreads) {
          const int32_t pj = tsorted[j];
          const uint32_t d = j + count_below(out, n_def, pj);
          if (d < (uint32_t)k) dst[d] = pj;
        }
        for (uint32_t i = n_def + nsel + threadIdx.x; i < (uint32_t)k; i += kFinThreads) dst[i] = -1;
        return;
      }
      for (uint32_t i = threadIdx.x; i < nsel; i += kFinThreads)
        if (n_def + i < (uint32_t)k) out[n_def + i] = tsel[i];
      if (threadIdx.x == 0) s_nout = min(n_def + nsel, (uint32_t)k);
      sort_out = true;
    } else if (dense) {
      for (uint32_t i = threadIdx.x; i < (uint32_t)k; i += kFinThreads) dst[i] = i < n_def ? out[i] : -1;
      return;
    }
  } else {
    // heavy exact ties at (t, t2): keys above bin t are taken and bin t is
    // resolved exactly over the whole list (keys outside bin t read as 0,
    // below every candidate key)
    for (uint32_t g = threadIdx.x; g < M; g += kFinThreads) {
      const uint2 c = ld_flat(g);
      if ((int)(c.x >> (32 - kHistBits)) > t) {
        const uint32_t slot = atomicAdd(&s_nout, 1u);
        if (slot < (uint32_t)k) out[slot] = (int32_t)c.y;
      }
    }
    const auto ld_bin = [&](uint32_t g) -> uint2 {
      uint2 c = ld_flat(g);
      if ((int)(c.x >> (32 - kHistBits)) != t) c.x = 0u;
      return c;
    };
    __syncthreads();
    resolve_exact(M, r, kHistBits, (uint32_t)t << (32 - kHistBits), ld_bin, k, out, s_nout, h, scratch);
    sort_out = true;
  }
  __syncthreads();
  const uint32_t nout = min(s_nout, (uint32_t)k);
  bool inverted = false;
  for (uint32_t i = threadIdx.x; i + 1 < nout; i += kFinThreads) inverted |= out[i] > out[i + 1];
  if (__syncthreads_or(sort_out && inverted)) {
    int n2 = (int)blockDim.x;
    while (n2 < k) n2 <<= 1;
    for (int i = threadIdx.x; i < n2; i += blockDim.x)
      if (i >= (int)nout) out[i] = 0x7FFFFFFF;
    __syncthreads();
    block_sort_asc(out, n2);
  }
  for (uint32_t i = threadIdx.x; i < (uint32_t)k; i += kFinThreads) dst[i] = i < nout ? out[i] : -1;
}

// Clears the leading `words` 16-byte words of a workspace (the histograms and
// counters) as a kernel, so the clear joins the chain of dependent launches.
__global__ void zero_kernel(uint4* __restrict__ p, int64_t words) {
  pdl_begin();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < words; i += (int64_t)gridDim.x * blockDim.x)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

// ---- block pool ---------------------------------------------------------------
// bmax[b][j] = max of scores[b][block*j .. block*j+block) within [0, n_visible[b]).
__global__ void block_max_kernel(const float* __restrict__ scores, int64_t n, const int32_t* __restrict__ n_visible,
                                 int32_t block, int64_t nb, float* __restrict__ bmax) {
  pdl_begin();
  const int b = blockIdx.y;
  int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= nb) return;
  int64_t nv = n_visible ? min((int64_t)n_visible[b], n) : n;
  float m = -INFINITY;
  for (int r = 0; r < block; ++r) {
    int64_t p = j * block + r;
    if (p < nv) {
      float s = scores[(int64_t)b * n + p];
      if (!isnan(s)) m = fmaxf(m, s);
    }
  }
  bmax[(int64_t)b * nb + j] = m;
}

__global__ void pool_expand_kernel(const int32_t* __restrict__ blocks, int32_t n_blocks, int32_t block,
                                   const int32_t* __restrict__ n_visible, int64_t n, int32_t* __restrict__ pool) {
  pdl_begin();
  const int b = blockIdx.y;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)n_blocks * block) return;
  int64_t nv = n_visible ? min((int64_t)n_visible[b], n) : n;
  int32_t blk = blocks[(int64_t)b * n_blocks + i / block];
  int64_t p = blk >= 0 ? (int64_t)blk * block + i % block : -1;
  pool[(int64_t)b * n_blocks * block + i] = (p >= 0 && p < nv) ? (int32_t)p : -1;
}

}  // namespace csa2

using namespace csa2;

int csa2_read_and_clear_topk_error(cudaStream_t s) {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_topk_error, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return CSA2_ERR_CUDA;
  if (cudaMemcpyToSymbolAsync(g_topk_error, &z, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return CSA2_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return CSA2_ERR_CUDA;
  return v;
}

static int64_t topk_chunk(int32_t B, int64_t n) {
  // aim for a few CTAs per SM across the whole batch
  int64_t target_ctas = 152 * 4;
  int64_t per_row = (target_ctas + B - 1) / B;
  int64_t chunk = (n + per_row - 1) / per_row;
  chunk = (chunk + 1023) / 1024 * 1024;
  if (chunk < 2048) chunk = 2048;
  return chunk;
}

// Opts the finalize kernel into its dynamic shared memory, once per device.
static int topk_finalize_attr() {
  static Csa2PerDeviceOnce optin;
  return csa2_smem_optin((const void*)topk_finalize_kernel, (int)kFinSmem, optin);
}

extern "C" size_t csa2_topk_workspace_size(int32_t B, int64_t n, int32_t k) {
  if (B <= 0 || n < 0 || k <= 0) return 0;
  return topk_ws_layout(B, n, k, nullptr, nullptr);
}

// Clears the histogram and counters of a Top-K workspace (a kernel enqueued on
// `stream`) and returns the per-row histogram [B][kTopkHistBins] that a
// producer of the scores may fill (the decode scan does it in its epilogue),
// and the per-row tile counters (zeroed too) it may claim its tiles from.
int csa2_topk_prepare(int32_t B, int64_t n, int32_t k, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream, uint32_t** hist, int32_t** scan_ctr, int32_t* scan_ctr_stride) {
  size_t need = topk_ws_layout(B, n, k, nullptr, nullptr);
  if (!workspace || workspace_bytes < need || !csa2_aligned(workspace, 256)) return CSA2_ERR_WORKSPACE;
  TopkWs ws;
  topk_ws_layout(B, n, k, &ws, (char*)workspace);
  const int64_t words = (int64_t)(topk_ws_zero_bytes(B) / 16);  // a multiple of 256 bytes
  if (words > 0)
    CSA2_LAUNCH_PDL(zero_kernel, dim3((unsigned)((words + 255) / 256 < 304 ? (words + 255) / 256 : 304)), dim3(256),
                    0, stream, (uint4*)workspace, words);
  if (hist) *hist = ws.hist;
  if (scan_ctr) *scan_ctr = &ws.cnt[0].scan_tiles;
  if (scan_ctr_stride) *scan_ctr_stride = (int32_t)(sizeof(RowCounters) / sizeof(int32_t));
  return CSA2_OK;
}

// Select + finalize over scores whose histogram is complete in the workspace.
int csa2_topk_from_hist(const float* scores, int32_t B, int64_t n, const int32_t* n_valid, const int32_t* positions,
                        int32_t k, int32_t* idx, void* workspace, cudaStream_t stream) {
  TopkWs ws;
  topk_ws_layout(B, n, k, &ws, (char*)workspace);
  dim3 grid((unsigned)ws.n_regions, (unsigned)B);
  if (positions)
    CSA2_LAUNCH_PDL(topk_select_kernel<true>, grid, dim3(kSelThreads), 0, stream, scores, n, n_valid, positions, k, ws);
  else
    CSA2_LAUNCH_PDL(topk_select_kernel<false>, grid, dim3(kSelThreads), 0, stream, scores, n, n_valid,
                    (const int32_t*)nullptr, k, ws);
  CSA2_CHECK_LAUNCH();
  int rc = topk_finalize_attr();
  if (rc) return rc;
  CSA2_LAUNCH_PDL(topk_finalize_kernel, dim3((unsigned)B), dim3(kFinThreads), kFinSmem, stream, n, k, ws, idx,
                  (int)(positions == nullptr));
  CSA2_CHECK_LAUNCH();
  return CSA2_OK;
}

int csa2_launch_topk(const float* scores, int32_t B, int64_t n, const int32_t* n_valid, const int32_t* positions,
                     int32_t k, int32_t* idx, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (B == 0) return CSA2_OK;
  int rc = csa2_topk_prepare(B, n, k, workspace, workspace_bytes, stream, nullptr, nullptr, nullptr);
  if (rc) return rc;
  TopkWs ws;
  topk_ws_layout(B, n, k, &ws, (char*)workspace);
  int64_t chunk = topk_chunk(B, n);
  if (!positions && chunk >= n && n > 0) {
    // a CTA per whole row: histogram and candidates in one pass over the scores
    CSA2_LAUNCH_PDL(topk_collect_kernel, dim3((unsigned)B), dim3(kSelThreads), 0, stream, scores, n, n_valid, k, ws);
    CSA2_CHECK_LAUNCH();
    int rc = topk_finalize_attr();
    if (rc) return rc;
    CSA2_LAUNCH_PDL(topk_finalize_kernel, dim3((unsigned)B), dim3(kFinThreads), kFinSmem, stream, n, k, ws, idx, 1);
    CSA2_CHECK_LAUNCH();
    return CSA2_OK;
  }
  int64_t chunks = n > 0 ? (n + chunk - 1) / chunk : 1;
  dim3 grid((unsigned)chunks, (unsigned)B);
  CSA2_LAUNCH_PDL(topk_hist_kernel, grid, dim3(kSelThreads), 0, stream, scores, n, n_valid, positions, chunk, k, ws);
  CSA2_CHECK_LAUNCH();
  return csa2_topk_from_hist(scores, B, n, n_valid, positions, k, idx, workspace, stream);
}

extern "C" int csa2_topk(const float* scores, int32_t B, int64_t n, const int32_t* n_valid,
                         const int32_t* positions, int32_t k, int32_t* idx, void* workspace,
                         size_t workspace_bytes, csa2_stream_t stream) {
  if (!scores || !idx || B < 0 || n < 0) return CSA2_ERR_INVALID_ARG;
  if (k <= 0 || k > CSA2_MAX_TOPK) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (n > 0x7FFFFFFFLL) return CSA2_ERR_UNSUPPORTED_SHAPE;
  return csa2_launch_topk(scores, B, n, n_valid, positions, k, idx, workspace, workspace_bytes,
                          (cudaStream_t)stream);
}

extern "C" int csa2_block_max(const float* scores, int32_t B, int64_t n, const int32_t* n_visible, int32_t block,
                              float* bmax, csa2_stream_t stream) {
  if (!scores || !bmax || B < 0 || n < 0 || block <= 0) return CSA2_ERR_INVALID_ARG;
  const int64_t nb = (n + block - 1) / block;
  if (B == 0 || nb == 0) return CSA2_OK;
  CSA2_LAUNCH_PDL(block_max_kernel, dim3((unsigned)((nb + 255) / 256), (unsigned)B), dim3(256), 0,
                  (cudaStream_t)stream, scores, n, n_visible, block, nb, bmax);
  return CSA2_OK;
}

extern "C" size_t csa2_block_pool_workspace_size(int32_t B, int64_t n, int32_t block, int32_t n_blocks) {
  if (B <= 0 || n < 0 || block <= 0 || n_blocks <= 0) return 0;
  int64_t nb = (n + block - 1) / block;
  size_t off = align_up((size_t)B * (size_t)(nb > 0 ? nb : 1) * 4, 256);
  off += align_up((size_t)B * n_blocks * 4, 256);
  off += topk_ws_layout(B, nb, n_blocks, nullptr, nullptr);
  return off;
}

// Pool from block maxima already in place: Top-n_blocks of the maxima, then the
// positions of the chosen blocks. `workspace` holds the chosen blocks and the
// Top-K scratch.
int csa2_launch_pool_from_bmax(const float* bmax, int32_t B, int64_t n, const int32_t* n_visible, int32_t block,
                               int32_t n_blocks, int32_t* pool, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
  if (B == 0) return CSA2_OK;
  const int64_t nb = (n + block - 1) / block;
  char* base = (char*)workspace;
  int32_t* blocks = (int32_t*)base;
  const size_t off = align_up((size_t)B * n_blocks * 4, 256);
  if (workspace_bytes < off) return CSA2_ERR_WORKSPACE;
  int rc = csa2_launch_topk(bmax, B, nb, nullptr, nullptr, n_blocks, blocks, base + off, workspace_bytes - off,
                            stream);
  if (rc) return rc;
  const int64_t total = (int64_t)n_blocks * block;
  dim3 g2((unsigned)((total + 255) / 256), (unsigned)B);
  CSA2_LAUNCH_PDL(pool_expand_kernel, g2, dim3(256), 0, stream, (const int32_t*)blocks, n_blocks, block, n_visible, n,
                  pool);
  return CSA2_OK;
}

int csa2_launch_block_pool(const float* scores, int32_t B, int64_t n, const int32_t* n_visible, int32_t block,
                           int32_t n_blocks, int32_t* pool, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
  if (B == 0) return CSA2_OK;
  size_t need = csa2_block_pool_workspace_size(B, n, block, n_blocks);
  if (!workspace || workspace_bytes < need || !csa2_aligned(workspace, 256)) return CSA2_ERR_WORKSPACE;
  int64_t nb = (n + block - 1) / block;
  char* base = (char*)workspace;
  float* bmax = (float*)base;
  size_t off = align_up((size_t)B * (size_t)(nb > 0 ? nb : 1) * 4, 256);
  if (nb > 0) {
    dim3 g1((unsigned)((nb + 255) / 256), (unsigned)B);
    CSA2_LAUNCH_PDL(block_max_kernel, g1, dim3(256), 0, stream, scores, n, n_visible, block, nb, bmax);
  }
  return csa2_launch_pool_from_bmax(bmax, B, n, n_visible, block, n_blocks, pool, base + off, workspace_bytes - off,
                                    stream);
}

extern "C" int csa2_block_pool(const float* scores, int32_t B, int64_t n, const int32_t* n_visible, int32_t block,
                               int32_t n_blocks, int32_t* pool, void* workspace, size_t workspace_bytes,
                               csa2_stream_t stream) {
  if (!scores || !pool || B < 0 || n < 0 || block <= 0 || n_blocks <= 0) return CSA2_ERR_INVALID_ARG;
  if (n_blocks > CSA2_MAX_TOPK || n > 0x7FFFFFFFLL) return CSA2_ERR_UNSUPPORTED_SHAPE;
  return csa2_launch_block_pool(scores, B, n, n_visible, block, n_blocks, pool, workspace, workspace_bytes,
                                (cudaStream_t)stream);
}

// ---- Top-K without allocation: scratch in a fixed device buffer ---------------
// The buffer is a file-scope device array; host code must not pass its name to
// a kernel (on the host it is only a stand-in symbol), so the device address is
// looked up once per device with cudaGetSymbolAddress and cached.
static __device__ __align__(256) unsigned char g_topk_static_scratch[CSA2_TOPK_STATIC_SCRATCH_BYTES];

static int topk_static_scratch_address(void** out) {
  constexpr int kMaxDevices = 64;
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CSA2_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topk_static_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return CSA2_ERR_CUDA;
    }
    addr[dev] = p;
  }
  *out = addr[dev];
  return CSA2_OK;
}

extern "C" int csa2_topk_static(const float* scores, int32_t B, int64_t n, const int32_t* n_valid,
                                const int32_t* positions, int32_t k, int32_t* idx, csa2_stream_t stream) {
  if (!scores || !idx || B < 0 || n < 0) return CSA2_ERR_INVALID_ARG;
  if (k <= 0 || k > CSA2_MAX_TOPK) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (n > 0x7FFFFFFFLL) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (B == 0) return CSA2_OK;
  if (topk_ws_layout(B, n, k, nullptr, nullptr) > (size_t)CSA2_TOPK_STATIC_SCRATCH_BYTES) return CSA2_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  int rc = topk_static_scratch_address(&ws);
  if (rc) return rc;
  return csa2_launch_topk(scores, B, n, n_valid, positions, k, idx, ws, CSA2_TOPK_STATIC_SCRATCH_BYTES,
                          (cudaStream_t)stream);
}
