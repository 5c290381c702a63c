// Exact top-k of 32-bit keys with ties to the lower index and the result
// written in ascending index order.  Used for the top-B history keys (keys =
// order-mapped scores) and for query subselection (keys = inverted
// order-mapped cosines, so the largest key is the least similar query).
//
// MSB-first radix select over 4 digits of 8 bits: each pass histograms the
// digit of the keys that still match the chosen prefix (warp-aggregated
// shared-memory atomics: a warp adds once per distinct digit, into one of 8
// sub-histograms so that warps whose keys share a digit do not all contend
// on one address), the sub-histograms are summed, then warp 0 finds the
// digit holding the k-th key with a shuffle scan.  After the last digit the
// exact k-th key theta is known, with r = the number of keys equal to theta
// that still have to be taken (the r lowest-index ones).  A final pass walks
// the keys in index order, one block-width at a time, and writes every key
// above theta plus the first r keys equal to theta.
//
// The pieces are used by a single block (block_radix_topk) and by a
// thread-block cluster that splits one row of keys across its CTAs and sums
// the histograms through distributed shared memory (topk.cu).
#pragma once

#include "common.cuh"

namespace quoka {

constexpr int kRadixSubHists = 8;

// Zero `nsub` x 256 counters.  Caller synchronises.
__device__ __forceinline__ void radix_zero(unsigned int* h, int count) {
  for (int i = threadIdx.x; i < count; i += blockDim.x) h[i] = 0;
}

// Histogram of digit (key >> shift) & dmask over keys i < n with (key & mask) == prefix.
// Keys of neighbouring positions usually share the digit (in the first pass
// nearly all keys do) or do not match the prefix at all, so each warp adds
// the lanes that share the first matching lane's digit with one atomic (a
// ballot) and only the remaining lanes add one by one.
template <typename KeyAt>
__device__ __forceinline__ void radix_hist(const KeyAt& key_at, int n, uint32_t prefix, uint32_t mask, int shift,
                                           unsigned int (*sub)[256], uint32_t dmask = 255u) {
  const int lane = threadIdx.x & 31;
  unsigned int* my_hist = sub[(threadIdx.x >> 5) & (kRadixSubHists - 1)];
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + threadIdx.x;
    uint32_t bin = 0xFFFFFFFFu;
    if (i < n) {
      const uint32_t u = key_at(i);
      if ((u & mask) == prefix) bin = (u >> shift) & dmask;
    }
    const unsigned valid = __ballot_sync(0xffffffffu, bin != 0xFFFFFFFFu);
    if (valid != 0u) {
      const int leader = __ffs(valid) - 1;
      const uint32_t lb = __shfl_sync(0xffffffffu, bin, leader);
      const unsigned same = __ballot_sync(0xffffffffu, bin == lb);
      if (lane == leader) atomicAdd(&my_hist[lb], (unsigned)__popc(same));
      else if (bin != 0xFFFFFFFFu && bin != lb) atomicAdd(&my_hist[bin], 1u);
    }
  }
}

// hist[b] = sum of the sub-histograms.  Caller synchronises before and after.
__device__ __forceinline__ void radix_reduce(unsigned int (*sub)[256], unsigned int* hist) {
  for (int b = threadIdx.x; b < 256; b += blockDim.x) {
    unsigned t = 0;
#pragma unroll
    for (int j = 0; j < kRadixSubHists; ++j) t += sub[j][b];
    hist[b] = t;
  }
}

// Warp 0 only: c[j] holds the count of bin 255 - 8*lane - j.  Finds the bin
// holding the need-th largest key and the rank of that key inside the bin.
__device__ __forceinline__ void radix_find_digit(const unsigned* c, int need, int* out_bin, int* out_need) {
  const int lane = threadIdx.x & 31;
  unsigned tot = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) tot += c[j];
  unsigned incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const unsigned excl = incl - tot;            // keys in higher bins than this lane's
  if (excl < (unsigned)need && (unsigned)need <= incl) {
    unsigned cum = excl;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (cum + c[j] >= (unsigned)need) {
        *out_bin = 255 - 8 * lane - j;
        *out_need = need - (int)cum;
        break;
      }
      cum += c[j];
    }
  }
}

// Index-ordered compaction of keys i < n: writes out[pos] = index_base + i for
// every key above theta and for the keys equal to theta whose global tie rank
// (ties0 + their rank here) is below r.  taken0 = selected keys before this
// range.  Stops once k keys are written.  scan: 32 ints of shared memory.
template <typename KeyAt>
__device__ __forceinline__ void radix_compact(const KeyAt& key_at, int n, uint32_t theta, int r, int taken0, int ties0,
                                              int k, int index_base, int32_t* __restrict__ out, int* scan) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  int taken = taken0, ties = ties0;   // block-uniform running totals
  for (int base = 0; base < n && taken < k; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const uint32_t u = i < n ? key_at(i) : 0u;
    const bool gt = i < n && u > theta;
    const bool eq = i < n && u == theta;
    const unsigned bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
    int total;
    const int packed = block_exclusive_scan(lane == 0 ? ((__popc(bg) << 16) | __popc(be)) : 0, scan, &total);
    const int pw = __shfl_sync(0xffffffffu, packed, 0);   // the warp's exclusive prefix (lane 0 holds it)
    const int gt_before = pw >> 16, eq_before = pw & 0xFFFF;
    const int tie_room = max(0, r - ties - eq_before);     // ties this warp may still take
    if (gt || eq) {
      const int eq_rank = __popc(be & lt);
      if (gt || eq_rank < tie_room) {
        const int pos = taken + gt_before + min(eq_before, max(0, r - ties)) + __popc(bg & lt) +
                        min(eq_rank, tie_room);
        out[pos] = index_base + i;
      }
    }
    const int gt_tot = total >> 16, eq_tot = total & 0xFFFF;
    taken += gt_tot + min(eq_tot, max(0, r - ties));
    ties += eq_tot;
  }
}

// ---- variants over keys cached in shared memory as uint4 (4 keys per
// thread per step, which gives each warp four independent chains).  keys4
// holds ceil(n / 4) vectors; entries at index >= n are ignored.

__device__ __forceinline__ void radix_hist_one(uint32_t bin, int lane, unsigned int* my_hist) {
  const unsigned valid = __ballot_sync(0xffffffffu, bin != 0xFFFFFFFFu);
  if (valid != 0u) {
    const int leader = __ffs(valid) - 1;
    const uint32_t lb = __shfl_sync(0xffffffffu, bin, leader);
    const unsigned same = __ballot_sync(0xffffffffu, bin == lb);
    if (lane == leader) atomicAdd(&my_hist[lb], (unsigned)__popc(same));
    else if (bin != 0xFFFFFFFFu && bin != lb) atomicAdd(&my_hist[bin], 1u);
  }
}

__device__ __forceinline__ void radix_hist4(const uint4* __restrict__ keys4, int n, uint32_t prefix, uint32_t mask,
                                            int shift, unsigned int (*sub)[256], uint32_t dmask = 255u) {
  const int lane = threadIdx.x & 31;
  unsigned int* my_hist = sub[(threadIdx.x >> 5) & (kRadixSubHists - 1)];
  const int nv = (n + 3) >> 2;
  for (int base = 0; base < nv; base += blockDim.x) {
    const int v = base + threadIdx.x;
    uint32_t b[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
    if (v < nv) {
      const uint4 q = keys4[v];
      const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (4 * v + j < n && (u[j] & mask) == prefix) b[j] = (u[j] >> shift) & dmask;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) radix_hist_one(b[j], lane, my_hist);
  }
}

// Index-ordered compaction (see radix_compact) with 4 consecutive keys per thread.
__device__ __forceinline__ void radix_compact4(const uint4* __restrict__ keys4, int n, uint32_t theta, int r,
                                               int taken0, int ties0, int k, int index_base,
                                               int32_t* __restrict__ out, int* scan) {
  const int lane = threadIdx.x & 31;
  const int nv = (n + 3) >> 2;
  int taken = taken0, ties = ties0;   // block-uniform running totals
  for (int base = 0; base < nv && taken < k; base += blockDim.x) {
    const int v = base + threadIdx.x;
    bool gt[4] = {false, false, false, false}, eq[4] = {false, false, false, false};
    if (v < nv) {
      const uint4 q = keys4[v];
      const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        gt[j] = 4 * v + j < n && u[j] > theta;
        eq[j] = 4 * v + j < n && u[j] == theta;
      }
    }
    const int my_gt = gt[0] + gt[1] + gt[2] + gt[3], my_eq = eq[0] + eq[1] + eq[2] + eq[3];
    int total;
    const int excl = block_exclusive_scan((my_gt << 16) | my_eq, scan, &total);  // per-thread, in index order
    const int gt_before = excl >> 16, eq_before = excl & 0xFFFF;
    int pos = taken + gt_before + min(eq_before, max(0, r - ties));
    int tie_rank = ties + eq_before;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (gt[j]) {
        out[pos++] = index_base + 4 * v + j;
      } else if (eq[j]) {
        if (tie_rank < r) out[pos++] = index_base + 4 * v + j;
        ++tie_rank;
      }
    }
    const int gt_tot = total >> 16, eq_tot = total & 0xFFFF;
    taken += gt_tot + min(eq_tot, max(0, r - ties));
    ties += eq_tot;
  }
  (void)lane;
}

struct RadixSelectShared {
  unsigned int sub[kRadixSubHists][256];
  unsigned int hist[256];
  int scan[32];
  int bin;
  int need;
};

// Whole-block top-k over keys i < n (k in [1, n]).  Every thread calls it.
template <typename KeyAt>
__device__ void block_radix_topk(const KeyAt& key_at, int n, int k, int32_t* __restrict__ out,
                                 RadixSelectShared& sm) {
  uint32_t prefix = 0, mask = 0;
  int need = k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    radix_zero(&sm.sub[0][0], kRadixSubHists * 256);
    __syncthreads();
    radix_hist(key_at, n, prefix, mask, shift, sm.sub);
    __syncthreads();
    radix_reduce(sm.sub, sm.hist);
    __syncthreads();
    if (threadIdx.x < 32) {
      unsigned c[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) c[j] = sm.hist[255 - 8 * threadIdx.x - j];
      radix_find_digit(c, need, &sm.bin, &sm.need);
    }
    __syncthreads();
    prefix |= (uint32_t)sm.bin << shift;
    mask |= 255u << shift;
    need = sm.need;
    __syncthreads();
  }
  radix_compact(key_at, n, prefix, need, 0, 0, k, 0, out, sm.scan);
}

// Whole-block top-k over keys cached in shared memory as uint4 (4 per thread per step).
__device__ inline void block_radix_topk4(const uint4* __restrict__ keys4, int n, int k, int32_t* __restrict__ out,
                                  RadixSelectShared& sm) {
  uint32_t prefix = 0, mask = 0;
  int need = k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    radix_zero(&sm.sub[0][0], kRadixSubHists * 256);
    __syncthreads();
    radix_hist4(keys4, n, prefix, mask, shift, sm.sub);
    __syncthreads();
    radix_reduce(sm.sub, sm.hist);
    __syncthreads();
    if (threadIdx.x < 32) {
      unsigned c[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) c[j] = sm.hist[255 - 8 * threadIdx.x - j];
      radix_find_digit(c, need, &sm.bin, &sm.need);
    }
    __syncthreads();
    prefix |= (uint32_t)sm.bin << shift;
    mask |= 255u << shift;
    need = sm.need;
    __syncthreads();
  }
  radix_compact4(keys4, n, prefix, need, 0, 0, k, 0, out, sm.scan);
}

}  // namespace quoka
