// Exact top-k of one row of 32-bit keys split across the CTAs of a
// thread-block cluster (ties to the lower index, output in ascending index
// order).  Used for the top-B history keys (topk.cu) and for query
// subselection (qsel.cu).
//
// CTA `rank` of the cluster owns keys [t0, t0 + n) of the row.  Each digit
// pass (radix_select.cuh) builds this CTA's histogram; after a cluster
// barrier every CTA sums the NC histograms through distributed shared memory
// and finds the digit.  At the end each CTA counts its keys above / equal to
// the threshold, reads the counts of the lower-ranked CTAs, and writes its
// selected positions at the right offsets.
#pragma once

#include <cooperative_groups.h>

#include "radix_select.cuh"

namespace quoka {

struct ClusterTopkShared {
  unsigned int sub[kRadixSubHists][256];
  unsigned int hist[2][256];   // this CTA's digit histogram by pass parity, read by the whole cluster
  unsigned int merged[256];    // the cluster's histogram of the current pass
  int counts[2];               // this CTA's keys above / equal to the threshold
  int scan[32];
  int bin, need, gt_base, eq_base;
};

// k in [1, row length).  keys4: this CTA's keys in shared memory (16-byte
// aligned) when `cache`, else key_at(i) yields key t0 + i.  Every thread of
// every CTA of the cluster calls it; it ends with a cluster barrier, so the
// CTA's shared memory outlives every remote read of it.
// hist12: NULL, or the whole row's histogram of the top 12 bits of the keys,
// counted where the keys were produced; the select then starts from that
// digit and needs three passes (8, 8 and 4 bits) instead of four of 8 bits.
template <int NC, typename KeyAt>
__device__ void cluster_radix_topk(cooperative_groups::cluster_group& cluster, bool cache, const uint4* keys4,
                                   const KeyAt& key_at, int n, int t0, int k, int32_t* __restrict__ out,
                                   ClusterTopkShared& sm, const unsigned* __restrict__ hist12 = nullptr) {
  const int rank = (int)cluster.block_rank();
  uint32_t prefix = 0, mask = 0;
  int need = k;
  if (hist12 != nullptr) {
    // the 12-bit digit holding the k-th largest key: bins in descending order, 8 per thread
    constexpr int kPer = 4096 / 512;
    static_assert(kPer * 512 == 4096, "512 threads take 8 bins each");
    unsigned c[kPer], tot = 0;
    const int hi = 4095 - kPer * (int)threadIdx.x;   // this thread's highest bin
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      c[j] = threadIdx.x < 512 ? hist12[hi - j] : 0u;
      tot += c[j];
    }
    int total;
    const int excl = block_exclusive_scan((int)tot, sm.scan, &total);   // keys in higher bins
    if (threadIdx.x < 512 && excl < need && need <= excl + (int)tot) {
      unsigned cum = (unsigned)excl;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        if (cum + c[j] >= (unsigned)need) {
          sm.bin = hi - j;
          sm.need = need - (int)cum;
          break;
        }
        cum += c[j];
      }
    }
    __syncthreads();
    prefix = (uint32_t)sm.bin << 20;
    mask = 0xFFF00000u;
    need = sm.need;
  }
  const int npass = hist12 != nullptr ? 3 : 4;
  for (int pass = 0; pass < npass; ++pass) {
    // digits: 8 bits at 24, 16, 8, 0; after the 12-bit start 8 bits at 12 and 4, then 4 bits at 0
    const int shift = hist12 != nullptr ? (pass == 0 ? 12 : pass == 1 ? 4 : 0) : 24 - 8 * pass;
    const uint32_t dmask = (hist12 != nullptr && pass == 2) ? 15u : 255u;
    const int buf = pass & 1;
    radix_zero(&sm.sub[0][0], kRadixSubHists * 256);
    __syncthreads();
    if (cache) radix_hist4(keys4, n, prefix, mask, shift, sm.sub, dmask);
    else radix_hist(key_at, n, prefix, mask, shift, sm.sub, dmask);
    __syncthreads();
    radix_reduce(sm.sub, sm.hist[buf]);
    cluster.sync();                       // every CTA's histogram of this pass is ready
    for (int b = threadIdx.x; b < 256; b += blockDim.x) {   // merge bin b across the cluster
      unsigned t = 0;
#pragma unroll
      for (int q = 0; q < NC; ++q) t += cluster.map_shared_rank(&sm.hist[buf][0], q)[b];
      sm.merged[b] = t;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      unsigned c[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) c[j] = sm.merged[255 - 8 * threadIdx.x - j];
      radix_find_digit(c, need, &sm.bin, &sm.need);
    }
    __syncthreads();
    prefix |= (uint32_t)sm.bin << shift;
    mask |= dmask << shift;
    need = sm.need;
    // hist[buf] is next written two passes later, after a cluster barrier every CTA
    // reaches only once it has finished reading this pass's histograms.
  }
  const uint32_t theta = prefix;
  const int r = need;
  int n_gt = 0, n_eq = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint32_t u = cache ? reinterpret_cast<const uint32_t*>(keys4)[i] : key_at(i);
    n_gt += u > theta;
    n_eq += u == theta;
  }
  int tot_gt, tot_eq;
  block_exclusive_scan(n_gt, sm.scan, &tot_gt);
  block_exclusive_scan(n_eq, sm.scan, &tot_eq);
  if (threadIdx.x == 0) {
    sm.counts[0] = tot_gt;
    sm.counts[1] = tot_eq;
  }
  cluster.sync();
  if (threadIdx.x == 0) {
    int gb = 0, eb = 0;
    for (int q = 0; q < rank; ++q) {
      const int* rc = cluster.map_shared_rank(&sm.counts[0], q);
      gb += rc[0];
      eb += rc[1];
    }
    sm.gt_base = gb;
    sm.eq_base = eb;
  }
  __syncthreads();
  const int gt_base = sm.gt_base, eq_base = sm.eq_base;
  if (cache)
    radix_compact4(keys4, n, theta, r, gt_base + min(eq_base, r), eq_base, k, t0, out, sm.scan);
  else
    radix_compact(key_at, n, theta, r, gt_base + min(eq_base, r), eq_base, k, t0, out, sm.scan);
  cluster.sync();                         // keep this CTA's shared memory alive for remote readers
}

}  // namespace quoka
