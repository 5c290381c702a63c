// Top-B history keys per KV head (QUOKA Explained, "From scores to a smaller
// KV set"; QUOKA paper summary, "Chunked Prefill with QUOKA").
//
// A thread-block cluster of 8 CTAs per KV head runs the cluster radix select
// of cluster_topk.cuh on the order-preserving 32-bit keys of the scores.  CTA
// r of the cluster owns the r-th contiguous eighth of the head's keys and
// caches them in shared memory (up to 40K keys per CTA; larger slices are
// re-read from global memory, where they are L2-resident right after the
// scoring kernel).  In the fused chunk path the scoring kernel has already
// counted the top 12 bits of every score (hist), so the select starts from
// that digit.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"
#include "cluster_topk.cuh"

namespace cg = cooperative_groups;

namespace quoka {

constexpr int kTopkCluster = 8;
constexpr int kTopkThreads = 512;
constexpr int kTopkSliceCap = 40 * 1024;   // keys per CTA cached in shared memory (160 KB)

__global__ void __cluster_dims__(kTopkCluster, 1, 1) __launch_bounds__(kTopkThreads)
    k_topk_cluster(const float* __restrict__ scores, int T_len, int B_e, int32_t* __restrict__ sel, int per,
                   int cache, const unsigned* __restrict__ hist) {
  pdl_launch_dependents();
  pdl_wait_for(scores, hist);
  extern __shared__ __align__(16) uint32_t keys_s[];
  __shared__ ClusterTopkShared sm;
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

  cluster_radix_topk<kTopkCluster>(cluster, cache != 0, keys4, key_at, n, t0, B_e, sel + (size_t)g * B_e, sm,
                                   hist != nullptr ? hist + (size_t)g * kScoreHistBins : nullptr);
}

__global__ void k_iota_rows(int32_t* __restrict__ sel, int rows, int n) {
  pdl_launch_dependents();
  pdl_wait();
  const size_t total = (size_t)rows * n;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x)
    sel[i] = (int32_t)(i % n);
}

cudaError_t launch_topk(const float* scores, int H_kv, int T_len, int B_e, int32_t* sel, cudaStream_t st,
                        const unsigned* hist) {
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
                 cache, hist);
  count_launches(1);
  return e;
}

}  // namespace quoka
