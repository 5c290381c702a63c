// Block-wide exact top-k of 32-bit keys with ties to the lower index and the
// result written in ascending index order.  Used for the top-B history keys
// (keys = order-mapped scores) and for query subselection (keys = inverted
// order-mapped cosines, so the largest key is the least similar query).
//
// MSB-first radix select over 4 digits of 8 bits: each pass histograms the
// digit of the keys that still match the chosen prefix (warp-aggregated
// shared-memory atomics: a warp adds once per distinct digit, into one of 8
// sub-histograms so that warps whose keys share a digit do not all contend
// on one address), the sub-histograms are summed, then warp 0 finds the
// digit holding the k-th key with a shuffle scan.  After the last
// digit the exact k-th key theta is known, with r = the number of keys equal
// to theta that still have to be taken (the r lowest-index ones).  A final
// pass walks the keys in index order, 1024 at a time, and writes every key
// above theta plus the first r keys equal to theta.
#pragma once

#include "common.cuh"

namespace quoka {

constexpr int kRadixSubHists = 8;

struct RadixSelectShared {
  unsigned int sub[kRadixSubHists][256];
  unsigned int hist[256];
  int scan[32];
  int bin;
  int need;
};

// key_at(i) returns the key of element i (i < n).  k in [1, n].  Every thread
// of the block must call this; blockDim.x must be a multiple of 32.
template <typename KeyAt>
__device__ void block_radix_topk(const KeyAt& key_at, int n, int k, int32_t* __restrict__ out,
                                 RadixSelectShared& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  uint32_t prefix = 0, mask = 0;
  int need = k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = threadIdx.x; i < kRadixSubHists * 256; i += blockDim.x) (&sm.sub[0][0])[i] = 0;
    __syncthreads();
    unsigned int* my_hist = sm.sub[warp & (kRadixSubHists - 1)];
    for (int base = 0; base < n; base += blockDim.x) {
      const int i = base + threadIdx.x;
      uint32_t bin = 0xFFFFFFFFu;
      if (i < n) {
        const uint32_t u = key_at(i);
        if ((u & mask) == prefix) bin = (u >> shift) & 255u;
      }
      const unsigned grp = __match_any_sync(0xffffffffu, bin);
      if (bin != 0xFFFFFFFFu && lane == __ffs(grp) - 1) atomicAdd(&my_hist[bin], (unsigned)__popc(grp));
    }
    __syncthreads();
    for (int b = threadIdx.x; b < 256; b += blockDim.x) {
      unsigned t = 0;
#pragma unroll
      for (int j = 0; j < kRadixSubHists; ++j) t += sm.sub[j][b];
      sm.hist[b] = t;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 255-8l .. 248-8l, highest first
      unsigned c[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = sm.hist[255 - 8 * lane - j];
        tot += c[j];
      }
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
            sm.bin = 255 - 8 * lane - j;
            sm.need = need - (int)cum;
            break;
          }
          cum += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= (uint32_t)sm.bin << shift;
    mask |= 255u << shift;
    need = sm.need;
    __syncthreads();
  }
  const uint32_t theta = prefix;
  const int r = need;
  const unsigned lt = (1u << lane) - 1u;
  int taken = 0, ties = 0;   // block-uniform running totals
  for (int base = 0; base < n && taken < k; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const uint32_t u = i < n ? key_at(i) : 0u;
    const bool gt = i < n && u > theta;
    const bool eq = i < n && u == theta;
    const unsigned bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
    int total;
    const int packed = block_exclusive_scan(lane == 0 ? ((__popc(bg) << 16) | __popc(be)) : 0, sm.scan, &total);
    const int pw = __shfl_sync(0xffffffffu, packed, 0);   // the warp's exclusive prefix (lane 0 holds it)
    const int gt_before = pw >> 16, eq_before = pw & 0xFFFF;
    const int tie_room = max(0, r - ties - eq_before);     // ties this warp may still take
    if (gt || eq) {
      const int eq_rank = __popc(be & lt);
      const bool sel = gt || eq_rank < tie_room;
      if (sel) {
        const int pos = taken + gt_before + min(eq_before, max(0, r - ties)) + __popc(bg & lt) +
                        min(eq_rank, tie_room);
        out[pos] = i;
      }
    }
    const int gt_tot = total >> 16, eq_tot = total & 0xFFFF;
    taken += gt_tot + min(eq_tot, max(0, r - ties));
    ties += eq_tot;
  }
  (void)nwarps;
}

}  // namespace quoka
