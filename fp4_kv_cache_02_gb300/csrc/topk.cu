// topk.cu -- Top-K selection and the hierarchical block pool.
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", section
// 2.3 (the indexer selects the Top-K entries for each query) and section 2.3.2
// with Figure 5 (each block of positions takes the maximum index score among
// its positions; the highest-scoring blocks form the candidate pool).
//
// Radix/threshold select on order-preserving 32-bit keys of the fp32 scores:
//   1. histogram of the top 11 key bits per row (shared-memory histogram per
//      CTA, flushed to a per-row global histogram; the decode scan can build
//      it in its epilogue);
//   2. every CTA finds the threshold bin t of its row (the bin in which the
//      running count from the top reaches k), then streams its slice: keys
//      above bin t are selected outright, keys inside bin t become candidates;
//   3. one CTA per row resolves bin t exactly on the remaining 21 key bits,
//      breaks exact ties by smaller position, sorts the k positions ascending
//      and writes them.
// The result does not depend on the order in which CTAs run.
#include "common.cuh"

#include <mutex>

namespace csa2 {

__device__ int g_topk_error = 0;

constexpr int kHistBits = kTopkHistBits;  // 11
constexpr int kHistBins = kTopkHistBins;  // 2048
constexpr int kSelThreads = 256;

struct RowCounters {
  uint32_t n_sel;      // positions appended to sel
  uint32_t n_cand;     // (key, position) pairs appended to cand
  uint32_t done;       // select CTAs of the row that finished streaming
  uint32_t hist_done;  // histogram CTAs of the row that flushed their counts
  int32_t t;           // threshold bin (-1: fewer candidates than k)
  uint32_t above;      // candidates in bins above t
  uint32_t pad[2];
};

struct TopkWs {
  uint32_t* hist;       // [B][4096]
  RowCounters* cnt;     // [B]
  int32_t* sel;         // [B][k]
  uint2* cand;          // [B][n]  (key, position)
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline size_t topk_ws_layout(int32_t B, int64_t n, int32_t k, TopkWs* ws, char* base) {
  size_t off = 0;
  size_t hist = off; off = align_up(off + (size_t)B * kHistBins * 4, 256);
  size_t cnt = off;  off = align_up(off + (size_t)B * sizeof(RowCounters), 256);
  size_t sel = off;  off = align_up(off + (size_t)B * k * 4, 256);
  size_t cand = off; off = align_up(off + (size_t)B * (size_t)(n > 0 ? n : 1) * 8, 256);
  if (ws) {
    ws->hist = (uint32_t*)(base + hist);
    ws->cnt = (RowCounters*)(base + cnt);
    ws->sel = (int32_t*)(base + sel);
    ws->cand = (uint2*)(base + cand);
  }
  return off;
}

__host__ __device__ inline size_t topk_ws_zero_bytes(int32_t B) {
  return align_up(align_up((size_t)B * kHistBins * 4, 256) + (size_t)B * sizeof(RowCounters), 256);
}

__device__ __forceinline__ bool load_candidate(const float* __restrict__ scores, const int32_t* __restrict__ positions,
                                               int64_t row_off, int64_t i, int64_t nv, uint32_t* key, int32_t* pos) {
  if (i >= nv) return false;
  float s = scores[row_off + i];
  int32_t p = positions ? positions[row_off + i] : (int32_t)i;
  if (p < 0 || !score_is_candidate(s)) return false;
  *key = score_key(s);
  *pos = p;
  return true;
}

__device__ int find_threshold_bin(const uint32_t* h, int nbins, uint32_t need, uint32_t* above_out,
                                  uint32_t* scratch);

// ---- pass 1: histogram of the top kHistBits key bits --------------------------
__global__ void __launch_bounds__(kSelThreads) topk_hist_kernel(
    const float* __restrict__ scores, int64_t n, const int32_t* __restrict__ n_valid,
    const int32_t* __restrict__ positions, int64_t chunk, int32_t k, TopkWs ws) {
  __shared__ uint32_t sh[kHistBins];
  const int b = blockIdx.y;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  const int64_t row_off = (int64_t)b * n;
  int64_t nv = n_valid ? min((int64_t)n_valid[b], n) : n;
  int64_t lo = (int64_t)blockIdx.x * chunk, hi = min(lo + chunk, nv);
  for (int64_t sub = lo; sub < hi; sub += (int64_t)kSelThreads * 16) {
    uint32_t key[16];
    uint32_t ok = 0;
#pragma unroll
    for (int e = 0; e < 16; ++e) {  // all loads of the sub-chunk in flight first
      const int64_t i = sub + (int64_t)e * kSelThreads + threadIdx.x;
      int32_t p;
      ok |= (uint32_t)(i < hi && load_candidate(scores, positions, row_off, i, nv, &key[e], &p)) << e;
    }
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if (ok & (1u << e)) atomicAdd(&sh[key[e] >> (32 - kHistBits)], 1u);
  }
  __syncthreads();
  uint32_t* gh = ws.hist + (size_t)b * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x)
    if (sh[i]) atomicAdd(&gh[i], sh[i]);
}

// Block-wide search, from the top bin down, for the first bin at which the
// running count reaches `need`. Returns the bin (-1 if the total is below
// `need`) and the count strictly above it. `h` has `nbins` entries in shared
// memory, nbins a multiple of blockDim.x (a multiple of 32); `scratch` holds
// blockDim.x + 2 words. Thread j owns bins [nbins-(j+1)*per, nbins-j*per); a
// warp-shuffle scan over the threads finds the owner of the crossing.
__device__ int find_threshold_bin(const uint32_t* h, int nbins, uint32_t need, uint32_t* above_out,
                                  uint32_t* scratch) {
  const int per = nbins / blockDim.x;
  const int j = threadIdx.x, lane = j & 31, warp = j >> 5, nwarps = blockDim.x >> 5;
  const int top = nbins - j * per;
  uint32_t local = 0;
  for (int i = 0; i < per; ++i) local += h[top - 1 - ((i + j) % per)];  // rotated: no bank conflicts
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

// Exact r-th largest among `count` 32-bit keys (in global memory, key field of
// uint2 or the `x` values of an int array transform), restricted to those whose
// top `fixed_bits` equal `prefix`. Radix passes over the remaining bits with
// `bits_per_pass` bits each. Returns the full threshold key; *r_left is how
// many keys equal to the threshold are still needed.
template <typename KeyFn>
__device__ uint32_t radix_select_desc(int count, uint32_t need, int fixed_bits, uint32_t prefix,
                                      KeyFn keyfn, uint32_t* hist /*kHistBins*/, uint32_t* scratch,
                                      uint32_t* r_left) {
  int done_bits = fixed_bits;
  while (done_bits < 32) {
    int pass_bits = min(kHistBits, 32 - done_bits);
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

// ---- pass 2: stream, select above the threshold bin, finalize in the last CTA --
// Each sub-chunk of kSelThreads x kPerThread scores is classified in registers;
// one block scan and one reservation atomic per output list place the
// selected positions (key above bin t) and the bin-t candidates.
constexpr int kPerThread = 16;
constexpr int kSmemCand = 4096;  // bin-t candidates finalized in shared memory up to this count

__global__ void __launch_bounds__(kSelThreads) topk_select_kernel(
    const float* __restrict__ scores, int64_t n, const int32_t* __restrict__ n_valid,
    const int32_t* __restrict__ positions, int64_t chunk, int32_t k, TopkWs ws) {
  __shared__ uint32_t h[kHistBins];
  __shared__ uint32_t scratch[kSelThreads + 8];
  __shared__ uint32_t s_base[2];
  const int b = blockIdx.y;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) h[i] = __ldcg(ws.hist + (size_t)b * kHistBins + i);
  __syncthreads();
  uint32_t above;
  const int t = find_threshold_bin(h, kHistBins, (uint32_t)k, &above, scratch);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    ws.cnt[b].t = t;
    ws.cnt[b].above = above;
  }
  const int64_t row_off = (int64_t)b * n;
  int64_t nv = n_valid ? min((int64_t)n_valid[b], n) : n;
  int64_t lo = (int64_t)blockIdx.x * chunk, hi = min(lo + chunk, nv);
  RowCounters* cnt = ws.cnt + b;
  int32_t* sel = ws.sel + (size_t)b * k;
  uint2* cand = ws.cand + (size_t)b * n;
  for (int64_t sub = lo; sub < hi; sub += (int64_t)kSelThreads * kPerThread) {
    uint32_t key[kPerThread];
    int32_t pos[kPerThread];
    uint32_t take = 0, keep = 0;
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int64_t i = sub + (int64_t)e * kSelThreads + threadIdx.x;
      const bool ok = i < hi && load_candidate(scores, positions, row_off, i, nv, &key[e], &pos[e]);
      const int digit = ok ? (int)(key[e] >> (32 - kHistBits)) : -2;
      take |= (uint32_t)(ok && digit > t) << e;
      keep |= (uint32_t)(ok && digit == t) << e;
    }
    uint32_t total;
    const uint32_t excl = block_exclusive_scan(__popc(take) | ((uint32_t)__popc(keep) << 16), &total, scratch);
    if (threadIdx.x == 0) {
      s_base[0] = (total & 0xFFFFu) ? atomicAdd(&cnt->n_sel, total & 0xFFFFu) : 0u;
      s_base[1] = (total >> 16) ? atomicAdd(&cnt->n_cand, total >> 16) : 0u;
    }
    __syncthreads();
    uint32_t st = s_base[0] + (excl & 0xFFFFu), sk = s_base[1] + (excl >> 16);
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      if (take & (1u << e)) {
        if (st < (uint32_t)k) sel[st] = pos[e];
        else record_error(&g_topk_error, CSA2_ERR_DEVICE);
        ++st;
      }
      if (keep & (1u << e)) {
        if (sk < (uint32_t)n) cand[sk] = make_uint2(key[e], (uint32_t)pos[e]);
        else record_error(&g_topk_error, CSA2_ERR_DEVICE);
        ++sk;
      }
    }
    __syncthreads();  // s_base is rewritten by the next sub-chunk
  }
}

// Resolves bin t exactly and writes one row: out[0..s_nout) already holds the
// positions whose key lies above bin t; the n_cand bin-t candidates are read
// through `ld`. Keys above the exact threshold key are taken; among keys equal
// to it, the smallest positions. The k positions are sorted ascending into dst
// (-1 padding). h has kHistBins words, scratch blockDim.x + 8.
template <typename LoadFn>
__device__ void finalize_row(int t, uint32_t above, uint32_t c_t, uint32_t n_cand, int32_t k, LoadFn ld,
                             int32_t* out, uint32_t& s_nout, uint32_t* h, uint32_t* scratch, int32_t* dst) {
  if (t >= 0) {
    uint32_t r = (uint32_t)k - above;  // still needed from bin t (1 <= r <= c_t)
    if (r >= n_cand || r >= c_t) {
      for (uint32_t i = threadIdx.x; i < n_cand; i += blockDim.x) {
        uint32_t slot = atomicAdd(&s_nout, 1u);
        if (slot < (uint32_t)k) out[slot] = (int32_t)ld(i).y;
      }
    } else {
      uint32_t r2;
      uint32_t T = radix_select_desc(
          (int)n_cand, r, kHistBits, ((uint32_t)t) << (32 - kHistBits),
          [&](int i) { return ld((uint32_t)i).x; }, h, scratch, &r2);
      // keys above T are all taken; among keys equal to T the r2 smallest
      // positions are taken (select on ~position, largest first)
      uint32_t n_eq = 0;
      {
        // count keys == T
        __shared__ uint32_t s_eq;
        if (threadIdx.x == 0) s_eq = 0;
        __syncthreads();
        uint32_t local = 0;
        for (uint32_t i = threadIdx.x; i < n_cand; i += blockDim.x) local += (ld(i).x == T);
        atomicAdd(&s_eq, local);
        __syncthreads();
        n_eq = s_eq;
        __syncthreads();
      }
      uint32_t P = 0xFFFFFFFFu, r3 = 0;
      bool all_eq = r2 >= n_eq;
      if (!all_eq) {
        // positions are >= 0, so ~position has bit 31 set: select the r2
        // largest ~position among keys == T
        P = radix_select_desc(
            (int)n_cand, r2, 0, 0u,
            [&](int i) {
              const uint2 c = ld((uint32_t)i);
              return c.x == T ? ~c.y : 0u;
            },
            h, scratch, &r3);
      }
      // keys above T, ties at T with ~position above P, and r3 of the ties
      // sitting exactly at ~position == P (a ticket; they share one position)
      __shared__ uint32_t s_r3;
      if (threadIdx.x == 0) s_r3 = 0;
      __syncthreads();
      for (uint32_t i = threadIdx.x; i < n_cand; i += blockDim.x) {
        const uint2 c = ld(i);
        bool take = c.x > T || (c.x == T && (all_eq || (~c.y) > P));
        if (!take && !all_eq && c.x == T && ~c.y == P) take = atomicAdd(&s_r3, 1u) < r3;
        if (take) {
          uint32_t slot = atomicAdd(&s_nout, 1u);
          if (slot < (uint32_t)k) out[slot] = (int32_t)c.y;
        }
      }
    }
  }
  __syncthreads();
  uint32_t nout = min(s_nout, (uint32_t)k);
  int n2 = (int)blockDim.x;
  while (n2 < k) n2 <<= 1;
  for (int i = threadIdx.x; i < n2; i += blockDim.x)
    if (i >= (int)nout) out[i] = 0x7FFFFFFF;
  __syncthreads();
  block_sort_asc(out, n2);
  for (int i = threadIdx.x; i < k; i += blockDim.x) dst[i] = i < (int)nout ? out[i] : -1;
}

// ---- pass 3: one CTA per row resolves bin t exactly and writes the row ------
__global__ void __launch_bounds__(kSelThreads) topk_finalize_kernel(int64_t n, int32_t k, TopkWs ws,
                                                                    int32_t* __restrict__ idx) {
  extern __shared__ uint32_t smem[];
  uint32_t* h = smem;                    // kHistBins
  uint32_t* scratch = smem + kHistBins;  // kSelThreads + 8
  int32_t* out = (int32_t*)(smem + kHistBins + kSelThreads + 8);                 // CSA2_MAX_TOPK
  uint2* cand_s = (uint2*)(smem + kHistBins + kSelThreads + 8 + CSA2_MAX_TOPK);  // kSmemCand
  __shared__ uint32_t s_nout;
  const int b = blockIdx.x;
  RowCounters* cnt = ws.cnt + b;
  const int32_t* sel = ws.sel + (size_t)b * k;
  const uint2* cand = ws.cand + (size_t)b * n;
  const int t = cnt->t;
  const uint32_t above = cnt->above;
  const uint32_t c_t = t >= 0 ? ws.hist[(size_t)b * kHistBins + t] : 0u;
  const uint32_t n_sel = min(cnt->n_sel, (uint32_t)k);
  const uint32_t n_cand = min(cnt->n_cand, (uint32_t)n);
  const bool in_smem = n_cand <= (uint32_t)kSmemCand;
  if (in_smem)
    for (uint32_t i = threadIdx.x; i < n_cand; i += blockDim.x) cand_s[i] = cand[i];
  for (uint32_t i = threadIdx.x; i < n_sel; i += blockDim.x) out[i] = sel[i];
  if (threadIdx.x == 0) s_nout = n_sel;
  __syncthreads();
  finalize_row(t, above, c_t, n_cand, k, [&](uint32_t i) -> uint2 { return in_smem ? cand_s[i] : cand[i]; }, out,
               s_nout, h, scratch, idx + (size_t)b * k);
}

// ---- block pool ---------------------------------------------------------------
// bmax[b][j] = max of scores[b][block*j .. block*j+block) within [0, n_visible[b]).
__global__ void block_max_kernel(const float* __restrict__ scores, int64_t n, const int32_t* __restrict__ n_visible,
                                 int32_t block, int64_t nb, float* __restrict__ bmax) {
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

static size_t topk_finalize_smem() {
  // histogram / radix scratch, the output list (up to CSA2_MAX_TOPK), kSmemCand candidates
  return (size_t)(kHistBins + kSelThreads + 8 + CSA2_MAX_TOPK) * 4 + (size_t)kSmemCand * 8;
}

extern "C" size_t csa2_topk_workspace_size(int32_t B, int64_t n, int32_t k) {
  if (B <= 0 || n < 0 || k <= 0) return 0;
  return topk_ws_layout(B, n, k, nullptr, nullptr);
}

// Clears the histogram and counters of a Top-K workspace (enqueued on
// `stream`) and returns the per-row histogram [B][kTopkHistBins] that a
// producer of the scores may fill (the decode scan does it in its epilogue).
int csa2_topk_prepare(int32_t B, int64_t n, int32_t k, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream, uint32_t** hist) {
  size_t need = topk_ws_layout(B, n, k, nullptr, nullptr);
  if (!workspace || workspace_bytes < need || !csa2_aligned(workspace, 256)) return CSA2_ERR_WORKSPACE;
  TopkWs ws;
  topk_ws_layout(B, n, k, &ws, (char*)workspace);
  if (cudaMemsetAsync(workspace, 0, topk_ws_zero_bytes(B), stream) != cudaSuccess) return CSA2_ERR_CUDA;
  if (hist) *hist = ws.hist;
  return CSA2_OK;
}

// Select + finalize over scores whose histogram is complete in the workspace.
int csa2_topk_from_hist(const float* scores, int32_t B, int64_t n, const int32_t* n_valid, const int32_t* positions,
                        int32_t k, int32_t* idx, void* workspace, cudaStream_t stream) {
  TopkWs ws;
  topk_ws_layout(B, n, k, &ws, (char*)workspace);
  int64_t chunk = topk_chunk(B, n);
  int64_t chunks = n > 0 ? (n + chunk - 1) / chunk : 1;
  dim3 grid((unsigned)chunks, (unsigned)B);
  topk_select_kernel<<<grid, kSelThreads, 0, stream>>>(scores, n, n_valid, positions, chunk, k, ws);
  CSA2_CHECK_LAUNCH();
  const size_t smem = topk_finalize_smem();
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(topk_finalize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return CSA2_ERR_CUDA;
    attr_set = true;
  }
  topk_finalize_kernel<<<(unsigned)B, kSelThreads, smem, stream>>>(n, k, ws, idx);
  CSA2_CHECK_LAUNCH();
  return CSA2_OK;
}

int csa2_launch_topk(const float* scores, int32_t B, int64_t n, const int32_t* n_valid, const int32_t* positions,
                     int32_t k, int32_t* idx, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (B == 0) return CSA2_OK;
  int rc = csa2_topk_prepare(B, n, k, workspace, workspace_bytes, stream, nullptr);
  if (rc) return rc;
  TopkWs ws;
  topk_ws_layout(B, n, k, &ws, (char*)workspace);
  int64_t chunk = topk_chunk(B, n);
  int64_t chunks = n > 0 ? (n + chunk - 1) / chunk : 1;
  dim3 grid((unsigned)chunks, (unsigned)B);
  topk_hist_kernel<<<grid, kSelThreads, 0, stream>>>(scores, n, n_valid, positions, chunk, k, ws);
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

extern "C" size_t csa2_block_pool_workspace_size(int32_t B, int64_t n, int32_t block, int32_t n_blocks) {
  if (B <= 0 || n < 0 || block <= 0 || n_blocks <= 0) return 0;
  int64_t nb = (n + block - 1) / block;
  size_t off = align_up((size_t)B * (size_t)(nb > 0 ? nb : 1) * 4, 256);
  off += align_up((size_t)B * n_blocks * 4, 256);
  off += topk_ws_layout(B, nb, n_blocks, nullptr, nullptr);
  return off;
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
  int32_t* blocks = (int32_t*)(base + off);
  off += align_up((size_t)B * n_blocks * 4, 256);
  if (nb > 0) {
    dim3 g1((unsigned)((nb + 255) / 256), (unsigned)B);
    block_max_kernel<<<g1, 256, 0, stream>>>(scores, n, n_visible, block, nb, bmax);
    CSA2_CHECK_LAUNCH();
  }
  int rc = csa2_launch_topk(bmax, B, nb, nullptr, nullptr, n_blocks, blocks, base + off, workspace_bytes - off,
                            stream);
  if (rc) return rc;
  int64_t total = (int64_t)n_blocks * block;
  dim3 g2((unsigned)((total + 255) / 256), (unsigned)B);
  pool_expand_kernel<<<g2, 256, 0, stream>>>(blocks, n_blocks, block, n_visible, n, pool);
  CSA2_CHECK_LAUNCH();
  return CSA2_OK;
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
