// Top-B history keys per KV head (QUOKA Explained, "From scores to a smaller
// KV set"; QUOKA paper summary, "Chunked Prefill with QUOKA").
//
// A thread-block cluster of 8 CTAs per KV head selects on the
// order-preserving 32-bit keys of the scores; CTA r of the cluster owns the
// r-th contiguous eighth of the head's keys and caches them in shared memory.
//
// In the fused chunk path the scoring kernel has already counted the top 12
// bits of every key (hist), and k_topk_fused needs two cluster barriers:
// every CTA finds the 12-bit bin b* that holds the B-th largest key, keeps the
// keys above it and lists its keys inside it (the candidates); CTA 0 gathers
// the candidates of the whole cluster over distributed shared memory, finds
// the exact threshold among them in two 10-bit radix passes, and pushes to
// every CTA its output offset and its share of the keys equal to the
// threshold (ties go to the lower position, and the CTAs own increasing
// positions); each CTA then writes its kept positions in ascending order.
// When the bin holds more candidates than CTA 0 can hold (many equal
// scores), every CTA runs the general select below instead.
//
// k_topk_cluster is the general select (cluster_topk.cuh): four 8-bit radix
// passes, or three after the 12-bit histogram, each with a cluster barrier
// (slices up to 40K keys per CTA in shared memory; larger slices are re-read
// from global memory, where they are L2-resident after the scoring kernel).
#include <cooperative_groups.h>

#include <algorithm>

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
  pdl_launch_dependents();   // dependents launch once this CTA is done
}

constexpr int kCandCap = 8192;   // candidates CTA 0 resolves in shared memory

struct FusedTopkShared {
  ClusterTopkShared general;     // the general select, when the bin is too full
  unsigned hist10[1024];         // CTA 0: 10-bit digit histogram of the candidates
  int gt[kTopkCluster], eq[kTopkCluster], def[kTopkCluster];   // CTA 0: per CTA of the cluster
  int scan[32];
  uint32_t bstar;                // the 12-bit bin of the B-th largest key
  int need;                      // keys to take from that bin
  int n_bin;                     // keys of the head in that bin
  int n_cand;                    // CTA 0: candidates pushed so far (by every CTA)
  int cand_base;                 // this CTA's first slot in CTA 0's candidate list
  int bin, bin_need;             // CTA 0: digit found by a pass
  uint32_t theta;                // pushed by CTA 0: the B-th largest key
  int quota, offset;             // pushed by CTA 0: this CTA's keys equal to theta to take, output offset
};

// Split cluster barrier: arrive (release) now, wait (acquire) later.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Shared-memory histogram add where the lanes of a warp with the same bin add once.
__device__ __forceinline__ void hist_add_warp(unsigned* hist, uint32_t bin, bool valid) {
  const uint32_t b = valid ? bin : 0xFFFFFFFFu;
  const unsigned peers = __match_any_sync(0xffffffffu, b);
  if (valid && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], (unsigned)__popc(peers));
}

// Block-wide: the bin of a 1024-bin histogram (descending order) holding the
// need-th largest key, and the rank of that key inside the bin.
__device__ __forceinline__ void find_desc_1024(const unsigned* h, int need, FusedTopkShared& sm) {
  const int i = threadIdx.x;                       // bins 1023 - 2i and 1022 - 2i
  const unsigned c0 = i < 512 ? h[1023 - 2 * i] : 0u, c1 = i < 512 ? h[1022 - 2 * i] : 0u;
  int total;
  const int excl = block_exclusive_scan((int)(c0 + c1), sm.scan, &total);
  if (i < 512 && excl < need && need <= excl + (int)(c0 + c1)) {
    if (need <= excl + (int)c0) {
      sm.bin = 1023 - 2 * i;
      sm.bin_need = need - excl;
    } else {
      sm.bin = 1022 - 2 * i;
      sm.bin_need = need - excl - (int)c0;
    }
  }
  __syncthreads();
}

__global__ void __cluster_dims__(kTopkCluster, 1, 1) __launch_bounds__(kTopkThreads)
    k_topk_fused(const float* __restrict__ scores, int T_len, int B_e, int32_t* __restrict__ sel, int per,
                 const unsigned* __restrict__ hist) {
  extern __shared__ __align__(16) uint32_t keys_s[];          // [per] this CTA's keys
  unsigned* h_s = keys_s + per;                                 // [4096] the head's 12-bit histogram
  uint2* gath = reinterpret_cast<uint2*>(h_s + kScoreHistBins); // [kCandCap] (key, position), CTA 0
  __shared__ FusedTopkShared sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int g = blockIdx.y;
  const int t0 = min(T_len, rank * per);
  const int n = min(T_len, t0 + per) - t0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* out = sel + (size_t)g * B_e;
  if (rank == 0 && threadIdx.x == 0) sm.n_cand = 0;
  cluster_arrive();            // CTA 0's counter is set before any CTA adds to it (waited for below)
  pdl_wait_for(scores, hist);
  const unsigned* h = hist + (size_t)g * kScoreHistBins;
  const float* s = scores + (size_t)g * T_len + t0;
  // the head's histogram and this CTA's keys into shared memory, all loads in flight together
  {
    const uint4* h4 = reinterpret_cast<const uint4*>(h);
    uint4 hv[kScoreHistBins / 4 / kTopkThreads];
#pragma unroll
    for (int j = 0; j < kScoreHistBins / 4 / kTopkThreads; ++j) hv[j] = h4[threadIdx.x + j * kTopkThreads];
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
#pragma unroll
    for (int j = 0; j < kScoreHistBins / 4 / kTopkThreads; ++j)
      reinterpret_cast<uint4*>(h_s)[threadIdx.x + j * kTopkThreads] = hv[j];
  }
  __syncthreads();
  if (warp == 0) {
    // the 12-bit bin holding the B_e-th largest key: lane l sums bins
    // [4096 - 128 (l + 1), 4096 - 128 l); a scan over the lanes (highest bins
    // first) finds the lane whose range crosses B_e, then the warp scans that
    // range 4 bins per lane
    unsigned tot = 0;
#pragma unroll 8
    for (int j = 0; j < 128; ++j) tot += h_s[kScoreHistBins - 128 * (lane + 1) + ((j + 4 * lane) & 127)];
    unsigned incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, incl - tot < (unsigned)B_e && (unsigned)B_e <= incl);
    const int L = __ffs(hit) - 1;                   // hit != 0: the bins sum to T >= B_e
    const unsigned above = __shfl_sync(0xffffffffu, incl - tot, L);
    const int hi = kScoreHistBins - 1 - 128 * L - 4 * lane;    // this lane's 4 bins: hi, hi - 1, hi - 2, hi - 3
    unsigned c[4], t4 = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      c[e] = h_s[hi - e];
      t4 += c[e];
    }
    unsigned in4 = t4;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(0xffffffffu, in4, o);
      if (lane >= o) in4 += y;
    }
    unsigned cum = above + in4 - t4;
    if (cum < (unsigned)B_e && (unsigned)B_e <= above + in4) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (cum < (unsigned)B_e && (unsigned)B_e <= cum + c[e]) {
          sm.bstar = (uint32_t)(hi - e);
          sm.need = B_e - (int)cum;
          sm.n_bin = (int)c[e];
        }
        cum += c[e];
      }
    }
  }
  __syncthreads();
  const uint4* keys4 = reinterpret_cast<const uint4*>(keys_s);
  if (sm.n_bin > kCandCap) {   // cluster-uniform: many keys in one bin, the general select
    cluster_wait();
    auto key_at = [&](int i) -> uint32_t { return keys_s[i]; };
    cluster_radix_topk<kTopkCluster>(cluster, true, keys4, key_at, n, t0, B_e, out, sm.general, h);
    return;
  }
  const uint32_t bstar = sm.bstar;
  // keys above the bin are kept; keys inside it are candidates, pushed to CTA 0 as (key, position)
  int my_def = 0, my_cand = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint32_t d = keys_s[i] >> 20;
    my_def += d > bstar;
    my_cand += d == bstar;
  }
  int n_def, n_cand;
  const int packed = block_exclusive_scan((my_cand << 16) | my_def, sm.scan, &n_def);
  n_cand = n_def >> 16;
  n_def &= 0xFFFF;
  cluster_wait();              // CTA 0's counter is initialised
  if (threadIdx.x == 0) {
    sm.cand_base = atomicAdd(cluster.map_shared_rank(&sm.n_cand, 0), n_cand);
    cluster.map_shared_rank(&sm, 0)->def[rank] = n_def;
  }
  __syncthreads();
  {
    uint2* dst = cluster.map_shared_rank(gath, 0);
    int at = sm.cand_base + (packed >> 16);
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const uint32_t k = keys_s[i];
      if ((k >> 20) == bstar && at < kCandCap) dst[at++] = make_uint2(k, (uint32_t)(t0 + i));
    }
  }
  cluster.sync();   // every candidate and count is in CTA 0

  if (rank == 0) {
    const int nc = min(sm.n_cand, kCandCap);   // equals the bin's count, which the branch above bounded
    for (int b = threadIdx.x; b < 1024; b += blockDim.x) sm.hist10[b] = 0;
    if (threadIdx.x < kTopkCluster) sm.gt[threadIdx.x] = sm.eq[threadIdx.x] = 0;
    __syncthreads();
    // two 10-bit passes over the candidates' low 20 bits
    for (int j0 = 0; j0 < nc; j0 += blockDim.x) {
      const int j = j0 + threadIdx.x;
      hist_add_warp(sm.hist10, j < nc ? (gath[j].x >> 10) & 1023u : 0u, j < nc);
    }
    __syncthreads();
    find_desc_1024(sm.hist10, sm.need, sm);
    const uint32_t dA = (uint32_t)sm.bin;
    const int needA = sm.bin_need;
    for (int b = threadIdx.x; b < 1024; b += blockDim.x) sm.hist10[b] = 0;
    __syncthreads();
    for (int j0 = 0; j0 < nc; j0 += blockDim.x) {
      const int j = j0 + threadIdx.x;
      const uint32_t k = j < nc ? gath[j].x : 0u;
      hist_add_warp(sm.hist10, k & 1023u, j < nc && ((k >> 10) & 1023u) == dA);
    }
    __syncthreads();
    find_desc_1024(sm.hist10, needA, sm);
    const uint32_t theta = (bstar << 20) | (dA << 10) | (uint32_t)sm.bin;
    const int r = sm.bin_need;                      // keys equal to theta to take, lowest positions first
    // per CTA: candidates above theta and equal to it
    for (int j0 = 0; j0 < nc; j0 += blockDim.x) {
      const int j = j0 + threadIdx.x;
      const uint2 c = j < nc ? gath[j] : make_uint2(0u, 0u);
      const int q = (int)(c.y / (uint32_t)per);
      hist_add_warp(reinterpret_cast<unsigned*>(sm.gt), (uint32_t)q, j < nc && c.x > theta);
      hist_add_warp(reinterpret_cast<unsigned*>(sm.eq), (uint32_t)q, j < nc && c.x == theta);
    }
    __syncthreads();
    if (threadIdx.x < kTopkCluster) {   // offsets and tie quotas, pushed to every CTA
      const int q = threadIdx.x;
      int off = 0, ties = 0;
      for (int p = 0; p < q; ++p) {
        off += sm.def[p] + sm.gt[p] + min(sm.eq[p], max(0, r - ties));
        ties += sm.eq[p];
      }
      FusedTopkShared* rs = cluster.map_shared_rank(&sm, q);
      rs->theta = theta;
      rs->quota = min(sm.eq[q], max(0, r - ties));
      rs->offset = off;
    }
  }
  cluster.sync();   // theta, quota and offset are in every CTA (no remote access after this)
  radix_compact4(keys4, n, sm.theta, sm.quota, sm.offset, 0, B_e, t0, out, sm.scan);
  pdl_launch_dependents();   // dependents launch once this CTA is done
}

__global__ void k_iota_rows(int32_t* __restrict__ sel, int rows, int n) {
  pdl_wait();
  const size_t total = (size_t)rows * n;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x)
    sel[i] = (int32_t)(i % n);
  pdl_launch_dependents();   // dependents launch once this CTA is done
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
  // at least 120 KB: one CTA per SM (two sharing an SM, as they do when they take SMs while the
  // scorer's CTAs finish, were 40% slower)
  const size_t fused_smem = std::max<size_t>((size_t)per * 4 + (size_t)kScoreHistBins * 4 + (size_t)kCandCap * 8,
                                             120 * 1024);
  cudaError_t e;
  if (hist != nullptr && fused_smem <= 200 * 1024) {
    if ((e = ensure_smem((const void*)k_topk_fused, fused_smem)) != cudaSuccess) return e;
    e = launch_pdl(k_topk_fused, dim3(kTopkCluster, H_kv), dim3(kTopkThreads), fused_smem, st, scores, T_len, B_e,
                   sel, per, hist);
    count_launches(1);
    return e;
  }
  const int cache = per <= kTopkSliceCap ? 1 : 0;
  const size_t smem = cache ? (size_t)per * 4 + 16 : 0;
  e = ensure_smem((const void*)k_topk_cluster, smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(k_topk_cluster, dim3(kTopkCluster, H_kv), dim3(kTopkThreads), smem, st, scores, T_len, B_e, sel, per,
                 cache, hist);
  count_launches(1);
  return e;
}

}  // namespace quoka
