// Exact top-k of one row of keys held by one CTA, from a 12-bit histogram.
//
// The keys are order-preserving 32-bit keys; bin_of maps a key to one of 4096
// bins and must be non-decreasing in the key (a coarse, monotone view of the
// value: fixed-point bins for cosines, or the key's top 12 bits).  The CTA
//   1. counts the bins (lanes of a warp with the same bin add once),
//   2. finds the bin b* holding the k-th largest key by one block scan,
//   3. lists the keys of b* (the candidates) with their positions,
//   4. finds the exact threshold key theta and the number r of keys equal to
//      it to keep: up to one candidate per thread by ranking every candidate
//      against the others, else by radix passes over the candidates' keys,
//   5. writes the positions of the keys above theta and of the first r equal
//      to it, ascending (ties go to the lower position).
// The candidate list has room for every key, so no distribution of values
// (equal keys included) needs another path.
#pragma once

#include "common.cuh"

namespace quoka {

constexpr int kBlockSelBins = 4096;

struct BlockSelectShared {
  alignas(16) unsigned hist[kBlockSelBins];   // the 12-bit histogram; later two 1024-bin digit histograms
  int scan[32];
  uint32_t bstar;    // the bin of the k-th largest key
  int need;          // keys to take from it
  int n_cand;
  int bin, bin_need;
  uint32_t theta;
  int r;
};

// One warp: the bin of a 1024-bin histogram (descending order) holding the
// need-th largest key, and that key's rank inside the bin.
__device__ __forceinline__ void block_select_find_1024(const unsigned* h, int need, BlockSelectShared& sm) {
  const int lane = threadIdx.x & 31;
  const uint4* h4 = reinterpret_cast<const uint4*>(h + 992 - 32 * lane);   // bins 1023 - 32 l .. 992 - 32 l
  unsigned c[32];
  int tot = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 v = h4[i];
    c[4 * i] = v.x;
    c[4 * i + 1] = v.y;
    c[4 * i + 2] = v.z;
    c[4 * i + 3] = v.w;
  }
#pragma unroll
  for (int e = 0; e < 32; ++e) tot += (int)c[e];
  int incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (incl - tot < need && need <= incl) {
    int cum = incl - tot;
#pragma unroll
    for (int e = 31; e >= 0; --e) {
      if (cum < need && need <= cum + (int)c[e]) {
        sm.bin = 992 - 32 * lane + e;
        sm.bin_need = need - cum;
      }
      cum += (int)c[e];
    }
  }
}

// The k largest of keys[0, n) (1 <= k <= n): out[0, k) receives index_base +
// their positions, ascending.  keys and cand (room for n pairs) are shared
// memory; every thread of the CTA calls it; blockDim.x is 256, 512 or 1024.
template <typename BinOf>
__device__ void block_select_top(const uint32_t* keys, int n, int k, int32_t* __restrict__ out, int index_base,
                                 uint2* cand, BlockSelectShared& sm, const BinOf& bin_of) {
  const int tid = threadIdx.x, nt = blockDim.x, warp = tid >> 5, lane = tid & 31;
  for (int b = tid; b < kBlockSelBins; b += nt) sm.hist[b] = 0u;
  if (tid == 0) {
    sm.n_cand = 0;
    sm.bstar = kBlockSelBins - 1;   // kept only if the bins do not sum to n (cannot happen)
    sm.need = k;
  }
  __syncthreads();
  // 1. the histogram
  for (int i0 = 0; i0 < n; i0 += nt) {
    const int i = i0 + tid;
    const bool v = i < n;
    hist_bin_add(sm.hist, v ? bin_of(keys[i]) : 0u, v);
  }
  __syncthreads();
  // 2. b*: thread t owns the bins 4095 - w t down to 4096 - w (t + 1), w = 4096 / blockDim.x
  {
    const int w = kBlockSelBins / nt;
    const int hi = kBlockSelBins - 1 - w * tid;
    int tot = 0;
    for (int j = 0; j < w; ++j) tot += (int)sm.hist[hi - j];
    int total;
    const int above = block_exclusive_scan(tot, sm.scan, &total);
    if (above < k && k <= above + tot) {
      int cum = above;
      for (int j = 0; j < w; ++j) {
        const int c = (int)sm.hist[hi - j];
        if (cum < k && k <= cum + c) {
          sm.bstar = (uint32_t)(hi - j);
          sm.need = k - cum;
        }
        cum += c;
      }
    }
    __syncthreads();
  }
  const uint32_t bstar = sm.bstar;
  // 3. the candidates (one shared counter add per warp and round)
  for (int i0 = 0; i0 < n; i0 += nt) {
    const int i = i0 + tid;
    const uint32_t key = i < n ? keys[i] : 0u;
    const bool c = i < n && bin_of(key) == bstar;
    const unsigned m = __ballot_sync(0xffffffffu, c);
    if (m != 0u) {
      const int leader = __ffs(m) - 1;
      int base = 0;
      if (lane == leader) base = atomicAdd(&sm.n_cand, __popc(m));
      base = __shfl_sync(0xffffffffu, base, leader);
      if (c) cand[base + __popc(m & ((1u << lane) - 1u))] = make_uint2(key, (uint32_t)i);
    }
  }
  __syncthreads();
  const int nc = sm.n_cand;
  // 4. theta and r
  if (nc <= nt) {
    if (tid < nc) {   // candidate tid: the keys above it and not below it
      const uint32_t ki = cand[tid].x;
      const int need = sm.need;
      int gt = 0, ge = 0;
      for (int j = 0; j < nc; ++j) {
        const uint32_t kj = cand[j].x;
        gt += kj > ki;
        ge += kj >= ki;
      }
      if (gt < need && need <= ge) {   // written alike by every candidate equal to theta
        sm.theta = ki;
        sm.r = need - gt;
      }
    }
    __syncthreads();
  } else {
    // radix passes of 10, 10, 10 and 2 bits over the candidates' keys (plain
    // shared atomics: a bin's keys spread over the digits)
    for (int b = tid; b < 2048; b += nt) sm.hist[b] = 0u;
    __syncthreads();
    uint32_t prefix = 0u;
    int pbits = 0, need = sm.need;
    for (int pass = 0; pbits < 32; ++pass) {
      const int width = min(10, 32 - pbits), shift = 32 - pbits - width;
      unsigned* h = sm.hist + 1024 * (pass & 1);
      for (int j = tid; j < nc; j += nt) {
        const uint32_t c = cand[j].x;
        if (pbits == 0 || (c >> (32 - pbits)) == prefix) atomicAdd(&h[(c >> shift) & ((1u << width) - 1u)], 1u);
      }
      __syncthreads();
      if (warp == 0) block_select_find_1024(h, need, sm);
      for (int b = tid; b < 1024; b += nt) sm.hist[1024 * ((pass + 1) & 1) + b] = 0u;   // the next pass's histogram
      __syncthreads();
      prefix = (prefix << width) | (uint32_t)sm.bin;
      pbits += width;
      need = sm.bin_need;
    }
    if (tid == 0) {
      sm.theta = prefix;
      sm.r = need;
    }
    __syncthreads();
  }
  const uint32_t theta = sm.theta;
  const int r = sm.r;
  // 5. thread t takes the positions kpt t .. kpt t + kpt - 1 (kpt odd: the
  //    threads' shared-memory reads fall in different banks)
  const int kpt = ((n + nt - 1) / nt) | 1;
  const int i0 = kpt * tid;
  int n_gt = 0, n_eq = 0;
  for (int j = 0; j < kpt; ++j) {
    const int i = i0 + j;
    if (i < n) {
      const uint32_t key = keys[i];
      n_gt += key > theta;
      n_eq += key == theta;
    }
  }
  int tot;
  const int ex = block_exclusive_scan((n_gt << 16) | n_eq, sm.scan, &tot);
  int gt_b = ex >> 16, eq_b = ex & 0xFFFF;
  if (n_gt + n_eq > 0) {
    for (int j = 0; j < kpt; ++j) {
      const int i = i0 + j;
      if (i >= n) break;
      const uint32_t key = keys[i];
      if (key > theta) {
        const int o = gt_b + min(eq_b, r);
        if (o < k) out[o] = index_base + i;
        ++gt_b;
      } else if (key == theta) {
        if (eq_b < r && gt_b + eq_b < k) out[gt_b + eq_b] = index_base + i;
        ++eq_b;
      }
    }
  }
}

}  // namespace quoka
