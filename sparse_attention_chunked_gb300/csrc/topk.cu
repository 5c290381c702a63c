// Top-B history keys per KV head (QUOKA Explained, "From scores to a smaller
// KV set"; QUOKA paper summary, "Chunked Prefill with QUOKA").
//
// A thread-block cluster of 8 CTAs per KV head runs an exact radix select
// (radix_select.cuh) on the order-preserving 32-bit keys of the scores.  CTA
// r of the cluster owns the r-th contiguous eighth of the head's keys and
// caches them in shared memory (up to 40K keys per CTA; larger slices are
// re-read from global memory, where they are L2-resident right after the
// scoring kernel).  Each digit pass builds per-CTA histograms; warp 0 of every
// CTA sums the 8 histograms through distributed shared memory and finds the
// digit.  At the end each CTA counts its keys above / equal to the threshold,
// reads the counts of the lower-ranked CTAs, and writes its selected positions
// at the right offsets, so the output is ascending and ties go to the lower
// position.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"
#include "radix_select.cuh"

namespace cg = cooperative_groups;

namespace quoka {

constexpr int kTopkCluster = 8;
constexpr int kTopkThreads = 512;
constexpr int kTopkSliceCap = 40 * 1024;   // keys per CTA cached in shared memory (160 KB)

struct TopkClusterShared {
  unsigned int sub[kRadixSubHists][256];
  unsigned int hist[2][256];   // this CTA's digit histogram by pass parity, read by the whole cluster
  unsigned int merged[256];    // the cluster's histogram of the current pass
  int counts[2];               // this CTA's keys above / equal to the threshold
  int scan[32];
  int bin, need, gt_base, eq_base;
};

__global__ void __cluster_dims__(kTopkCluster, 1, 1) __launch_bounds__(kTopkThreads)
    k_topk_cluster(const float* __restrict__ scores, int T_len, int B_e, int32_t* __restrict__ sel, int per,
                   int cache) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ __align__(16) uint32_t keys_s[];
  __shared__ TopkClusterShared sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int g = blockIdx.y;
  const int t0 = min(T_len, rank * per);
  const int n = min(T_len, t0 + per) - t0;
  const float* s = scores + (size_t)g * T_len + t0;
  if (cache) {
    // batched loads: 4 independent scores per thread in flight
    for (int i0 = threadIdx.x; i0 < n; i0 += 4 * blockDim.x) {
      float f[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + j * blockDim.x;
        f[j] = i < n ? s[i] : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + j * blockDim.x;
        if (i < n) keys_s[i] = order_key(f[j]);
      }
    }
    __syncthreads();
  }
  auto key_at = [&](int i) -> uint32_t { return cache ? keys_s[i] : order_key(s[i]); };
  const uint4* keys4 = reinterpret_cast<const uint4*>(keys_s);

  uint32_t prefix = 0, mask = 0;
  int need = B_e;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass, buf = pass & 1;
    radix_zero(&sm.sub[0][0], kRadixSubHists * 256);
    __syncthreads();
    if (cache) radix_hist4(keys4, n, prefix, mask, shift, sm.sub);
    else radix_hist(key_at, n, prefix, mask, shift, sm.sub);
    __syncthreads();
    radix_reduce(sm.sub, sm.hist[buf]);
    cluster.sync();                       // every CTA's histogram of this pass is ready
    for (int b = threadIdx.x; b < 256; b += blockDim.x) {   // merge bin b across the cluster
      unsigned t = 0;
#pragma unroll
      for (int q = 0; q < kTopkCluster; ++q) t += cluster.map_shared_rank(&sm.hist[buf][0], q)[b];
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
    mask |= 255u << shift;
    need = sm.need;
    // hist[buf] is next written two passes later, after a cluster barrier every CTA
    // reaches only once it has finished reading this pass's histograms.
  }
  const uint32_t theta = prefix;
  const int r = need;
  int n_gt = 0, n_eq = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint32_t u = key_at(i);
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
    radix_compact4(keys4, n, theta, r, gt_base + min(eq_base, r), eq_base, B_e, t0, sel + (size_t)g * B_e, sm.scan);
  else
    radix_compact(key_at, n, theta, r, gt_base + min(eq_base, r), eq_base, B_e, t0, sel + (size_t)g * B_e, sm.scan);
  cluster.sync();                         // keep this CTA's shared memory alive for remote readers
}

__global__ void k_iota_rows(int32_t* __restrict__ sel, int rows, int n) {
  pdl_launch_dependents();
  pdl_wait();
  const size_t total = (size_t)rows * n;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x)
    sel[i] = (int32_t)(i % n);
}

cudaError_t launch_topk(const float* scores, int H_kv, int T_len, int B_e, int32_t* sel, cudaStream_t st) {
  if (B_e == 0) return cudaSuccess;
  if (B_e >= T_len) {
    const size_t total = (size_t)H_kv * T_len;
    const size_t nb = (total + 255) / 256;
    const int blocks = (int)(nb < 4096 ? (nb == 0 ? 1 : nb) : 4096);
    cudaError_t e = launch_pdl(k_iota_rows, dim3(blocks), dim3(256), 0, st, sel, H_kv, T_len);
    count_launches(1);
    return e;
  }
  const int per = ((T_len + kTopkCluster - 1) / kTopkCluster + 3) & ~3;
  const int cache = per <= kTopkSliceCap ? 1 : 0;
  const size_t smem = cache ? (size_t)per * 4 + 16 : 0;
  cudaError_t e = ensure_smem((const void*)k_topk_cluster, smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(k_topk_cluster, dim3(kTopkCluster, H_kv), dim3(kTopkThreads), smem, st, scores, T_len, B_e, sel, per,
                 cache);
  count_launches(1);
  return e;
}

}  // namespace quoka
