// Top-B history keys per KV head (QUOKA Explained, "From scores to a smaller
// KV set"; QUOKA paper summary, "Chunked Prefill with QUOKA").
//
// A thread-block cluster of 8 CTAs per KV head selects on the
// order-preserving 32-bit keys of the scores; CTA r of the cluster owns the
// r-th contiguous eighth of the head's keys.
//
// In the fused chunk path the scoring kernel has already counted the top 12
// bits of every key, and k_topk_fused needs one cluster barrier (described at
// the kernel).  k_topk_cluster is the general select (cluster_topk.cuh): four
// 8-bit radix passes, or three after the 12-bit histogram, each with a
// cluster barrier (slices up to 40K keys per CTA in shared memory; larger
// slices are re-read from global memory, where they are L2-resident after the
// scoring kernel).  Ties go to the lower position, and the output is
// ascending.
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

constexpr int kCandCap = 12288;   // candidates, copied into every CTA of the cluster (96 KB)
constexpr int kStageCap = 4096;   // one CTA's own candidates, staged before the copy (32 KB)
constexpr int kFusedSliceCap = 16384;   // keys per CTA of the fused select (64 KB of shared memory)

struct FusedTopkShared {
  ClusterTopkShared general;     // the general select, when the list would overflow
  alignas(16) unsigned hist10[2][1024];   // 10-bit digit histograms of the candidates (bits 19-10,
                                          // 9-0), read as uint4
  int def_of[kTopkCluster];      // pushed by CTA q: its keys above the bin b*
  int cand_of[kTopkCluster];     // pushed by CTA q: its keys inside b*
  int red[kTopkThreads / 32][3];
  int scan[32];
  uint32_t bstar;                // the 12-bit bin of the B-th largest key
  int need;                      // keys to take from that bin
  int n_cand;                    // CTA 0: candidate slots handed out
  int cand_base;                 // this CTA's first candidate slot
  int bin, bin_need;             // digit found by a pass
  uint32_t theta;                // the B-th largest key
  int r;                         // keys equal to theta to keep
};

static_assert(offsetof(FusedTopkShared, hist10) % 16 == 0, "16-byte loads of the digit histograms");

// Split cluster barrier: arrive (release) now, wait (acquire) later.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// One warp: the bin of a 1024-bin histogram (descending order) holding the
// need-th largest key, and the rank of that key inside the bin.  Lane l sums
// bins 1023 - 32 l down to 992 - 32 l; a warp scan finds the lane whose range
// holds the key, and that lane walks its 32 bins.
__device__ __forceinline__ void warp_find_desc_1024(const unsigned* h, int need, FusedTopkShared& sm) {
  const int lane = threadIdx.x & 31;
  const uint4* h4 = reinterpret_cast<const uint4*>(h + 992 - 32 * lane);
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

// The key a score is selected on: order_key, with NaN as -inf where the bins
// are the fixed-point cosine bins (which count NaN in bin 0).
__device__ __forceinline__ uint32_t select_key(float f, bool cosine) {
  return order_key((cosine && f != f) ? -INFINITY : f);
}

constexpr int kRankMax = 128;   // candidates ranked directly (one per thread, against every other)

// The fused select (the scorer has counted a 12-bit histogram of its scores,
// score_bin).  CTA r of the cluster owns positions [r per, (r + 1) per) of the
// head, loads their keys into shared memory, and thread t of it takes the kpt
// consecutive positions from kpt t (kpt = per / 512 rounded up to a multiple
// of 4).  Every CTA finds the bin b* of the B-th largest score from the
// histogram, counts its keys above b* and lists its keys inside b* (the
// candidates, with their positions) in shared memory; it takes a range of
// slots from an atomic counter in CTA 0 and copies its list, with coalesced
// stores, to those slots of the candidate list of EVERY CTA of the cluster.
// After the one cluster barrier each CTA holds the whole candidate list and
// every CTA's counts, and finds on its own the exact threshold key theta (up
// to 128 candidates by ranking each against all others, else by radix passes
// over the candidates' keys), the number r of keys equal to theta to keep
// (lowest positions first), and its output offset: the kept keys of the lower
// ranks.  It then writes its kept positions in ascending order.  No shared
// memory is touched remotely after the barrier.  A list that would overflow
// (many equal scores) sends every CTA to the general select.  The per-key
// loops run over groups of 4 keys and are not unrolled: the kernel runs its
// code once per launch, and straight-line code for 32 keys per thread spent
// its time fetching instructions.
__global__ void __cluster_dims__(kTopkCluster, 1, 1) __launch_bounds__(kTopkThreads)
    k_topk_fused(const float* __restrict__ scores, int T_len, int B_e, int32_t* __restrict__ sel, int per,
                 const unsigned* __restrict__ hist, int vec, int cosine) {
  extern __shared__ __align__(16) uint2 cand[];   // [kCandCap] (key, position), [kStageCap] staged, [per] keys
  uint2* stage = cand + kCandCap;
  uint32_t* keys = reinterpret_cast<uint32_t*>(stage + kStageCap);
  const uint4* keys4 = reinterpret_cast<const uint4*>(keys);
  __shared__ FusedTopkShared sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y;
  const int t0 = min(T_len, rank * per);
  const int n = min(T_len, t0 + per) - t0;
  int32_t* out = sel + (size_t)g * B_e;
  sm.hist10[0][tid] = sm.hist10[0][tid + kTopkThreads] = 0u;
  if (tid == 0) {
    sm.n_cand = 0;
    sm.bstar = 0xFFFu;   // kept only if the histogram does not sum to T (cannot happen)
    sm.need = B_e;
  }
  cluster_arrive();      // CTA 0's counter is set before any CTA adds to it (waited for below)
  pdl_wait_for(scores, hist);
  const unsigned* h = hist + (size_t)g * kScoreHistBins;
  const float* s = scores + (size_t)g * T_len + t0;
  const uint4 ha = reinterpret_cast<const uint4*>(h)[1023 - 2 * tid];   // bins 4095 - 8t - 3 .. 4095 - 8t
  const uint4 hb = reinterpret_cast<const uint4*>(h)[1022 - 2 * tid];   // bins 4095 - 8t - 7 .. 4095 - 8t - 4
  // the slice's keys into shared memory (positions past n read as key 0 and are never counted)
  const int n4 = (n + 3) >> 2;
  if (vec) {   // T a multiple of 4 and 16-byte aligned rows
#pragma unroll 4
    for (int i = tid; i < n4; i += kTopkThreads) {
      const float4 f = reinterpret_cast<const float4*>(s)[i];
      reinterpret_cast<uint4*>(keys)[i] =
          make_uint4(select_key(f.x, cosine), select_key(f.y, cosine), select_key(f.z, cosine), select_key(f.w, cosine));
    }
  } else {
    for (int i = tid; i < 4 * n4; i += kTopkThreads) keys[i] = i < n ? select_key(s[i], cosine) : 0u;
  }
  // the 12-bit bin holding the B-th largest key: 8 bins per thread, descending
  {
    const int c[8] = {(int)ha.w, (int)ha.z, (int)ha.y, (int)ha.x, (int)hb.w, (int)hb.z, (int)hb.y, (int)hb.x};
    int tot = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) tot += c[j];
    int total;
    const int above = block_exclusive_scan(tot, sm.scan, &total);   // its barriers also publish the keys
    if (above < B_e && B_e <= above + tot) {
      int cum = above;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (cum < B_e && B_e <= cum + c[j]) {
          sm.bstar = (uint32_t)(kScoreHistBins - 1 - 8 * tid - j);
          sm.need = B_e - cum;
        }
        cum += c[j];
      }
    }
    __syncthreads();
  }
  const uint32_t bstar = sm.bstar;
  auto bin_of = [&](uint32_t key) -> uint32_t { return cosine ? score_bin(key_float(key), true) : key >> 20; };
  // this thread's keys: positions i0 .. i0 + kpt - 1 of the slice, 4 at a time
  const int kpt = ((per + kTopkThreads - 1) / kTopkThreads + 3) & ~3;
  const int i0 = kpt * tid;
  const int nv = max(0, min(kpt, n - i0));
  const int ng = (nv + 3) >> 2;
  int my_def = 0, my_cand = 0;
#pragma unroll 1
  for (int q = 0; q < ng; ++q) {
    const uint4 v = keys4[(i0 >> 2) + q];
    const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool ok = 4 * q + e < nv;
      const uint32_t d = bin_of(kk[e]);
      my_def += ok && d > bstar;
      my_cand += ok && d == bstar;
    }
  }
  int tot_packed;
  const int excl = block_exclusive_scan((my_cand << 16) | my_def, sm.scan, &tot_packed);
  const int n_def = tot_packed & 0xFFFF, n_own = tot_packed >> 16;
  if (my_cand > 0) {   // this CTA's candidates, in position order
    int at = excl >> 16;
#pragma unroll 1
    for (int q = 0; q < ng; ++q) {
      const uint4 v = keys4[(i0 >> 2) + q];
      const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (4 * q + e < nv && bin_of(kk[e]) == bstar) {
          if (at < kStageCap) stage[at] = make_uint2(kk[e], (uint32_t)(t0 + i0 + 4 * q + e));
          ++at;
        }
      }
    }
  }
  cluster_wait();        // every CTA has started: CTA 0's counter is initialised
  if (tid == 0) sm.cand_base = atomicAdd(cluster.map_shared_rank(&sm.n_cand, 0), n_own);
  __syncthreads();       // the slot range and the staged list
  const int base = sm.cand_base;
  if (tid < kTopkCluster) {
    FusedTopkShared* rs = cluster.map_shared_rank(&sm, tid);
    rs->def_of[rank] = n_def;
    rs->cand_of[rank] = n_own;
  }
  {
    const int m = min(n_own, min(kStageCap, kCandCap - min(base, kCandCap)));
#pragma unroll 1
    for (int q = 0; q < kTopkCluster; ++q) {
      uint2* rc = cluster.map_shared_rank(cand, q) + base;
      for (int i = tid; i < m; i += kTopkThreads) rc[i] = stage[i];
    }
  }
  cluster.sync();        // every candidate and count is in every CTA; no remote access after this
  int nc = 0;
  bool overflow = false;
#pragma unroll
  for (int q = 0; q < kTopkCluster; ++q) {
    nc += sm.cand_of[q];
    overflow |= sm.cand_of[q] > kStageCap;
  }
  if (overflow || nc > kCandCap) {   // cluster-uniform: the general select on the keys in shared memory
    auto key_at = [&](int i) -> uint32_t { return keys[i]; };
    cluster_radix_topk<kTopkCluster>(cluster, true, keys4, key_at, n, t0, B_e, out, sm.general,
                                     cosine ? nullptr : h);
    return;
  }
  // theta and r
  if (nc <= kRankMax) {
    if (tid < nc) {   // candidate tid: keys above it and not below it
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
    // radix passes over the candidates' keys, 10 bits at a time below the
    // bits they share (the 12-bit bin, for order-key bins; none for cosine
    // bins).  The keys of one bin spread over the digits, so plain shared
    // atomics rarely collide.
    uint32_t prefix = cosine ? 0u : bstar;
    int pbits = cosine ? 0 : 12, need = sm.need;
    for (int pass = 0; pbits < 32; ++pass) {
      const int width = min(10, 32 - pbits), shift = 32 - pbits - width;
      unsigned* hh = sm.hist10[pass & 1];
      for (int j = tid; j < nc; j += kTopkThreads) {
        const uint32_t c = cand[j].x;
        if (pbits == 0 || (c >> (32 - pbits)) == prefix) atomicAdd(&hh[(c >> shift) & ((1u << width) - 1u)], 1u);
      }
      __syncthreads();
      if (warp == 0) warp_find_desc_1024(hh, need, sm);
      // the other histogram, used by the next pass, is cleared meanwhile
      sm.hist10[(pass + 1) & 1][tid] = sm.hist10[(pass + 1) & 1][tid + kTopkThreads] = 0u;
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
  const int r = sm.r;   // keys equal to theta to keep, lowest positions first
  // the keys of the lower ranks above and equal to theta, and this CTA's ties:
  // candidates at positions below t0, and inside [t0, t0 + n)
  int offset, quota;
  {
    int gt_lo = 0, eq_lo = 0, eq_me = 0;
    for (int j = tid; j < nc; j += kTopkThreads) {
      const uint2 c = cand[j];
      const bool lo = c.y < (uint32_t)t0;
      gt_lo += lo && c.x > theta;
      eq_lo += lo && c.x == theta;
      eq_me += !lo && c.y < (uint32_t)(t0 + n) && c.x == theta;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      gt_lo += __shfl_xor_sync(0xffffffffu, gt_lo, o);
      eq_lo += __shfl_xor_sync(0xffffffffu, eq_lo, o);
      eq_me += __shfl_xor_sync(0xffffffffu, eq_me, o);
    }
    if (lane == 0) {
      sm.red[warp][0] = gt_lo;
      sm.red[warp][1] = eq_lo;
      sm.red[warp][2] = eq_me;
    }
    __syncthreads();
    gt_lo = eq_lo = eq_me = 0;
#pragma unroll
    for (int w = 0; w < kTopkThreads / 32; ++w) {
      gt_lo += sm.red[w][0];
      eq_lo += sm.red[w][1];
      eq_me += sm.red[w][2];
    }
    int def_lo = 0;
#pragma unroll
    for (int q = 0; q < kTopkCluster; ++q) def_lo += q < rank ? sm.def_of[q] : 0;
    offset = def_lo + gt_lo + min(eq_lo, r);
    quota = min(eq_me, max(0, r - eq_lo));
  }
  // this CTA's kept positions, ascending: a key above theta goes after the keys
  // above theta before it and the kept ties before it
  int n_gt = 0, n_eq = 0;
#pragma unroll 1
  for (int q = 0; q < ng; ++q) {
    const uint4 v = keys4[(i0 >> 2) + q];
    const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool ok = 4 * q + e < nv;
      n_gt += ok && kk[e] > theta;
      n_eq += ok && kk[e] == theta;
    }
  }
  int tot2;
  const int ex2 = block_exclusive_scan((n_gt << 16) | n_eq, sm.scan, &tot2);
  int gt_b = ex2 >> 16, eq_b = ex2 & 0xFFFF;
  if (n_gt + n_eq > 0) {
#pragma unroll 1
    for (int q = 0; q < ng; ++q) {
      const uint4 v = keys4[(i0 >> 2) + q];
      const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (4 * q + e >= nv) continue;
        const int pos = t0 + i0 + 4 * q + e;
        if (kk[e] > theta) {
          const int o = offset + gt_b + min(eq_b, quota);
          if (o < B_e) out[o] = pos;
          ++gt_b;
        } else if (kk[e] == theta) {
          if (eq_b < quota && offset + gt_b + eq_b < B_e) out[offset + gt_b + eq_b] = pos;
          ++eq_b;
        }
      }
    }
  }
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
                        const unsigned* hist, bool cosine_bins) {
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
  cudaError_t e;
  if (hist != nullptr && per <= kFusedSliceCap) {
    // at least 120 KB of shared memory: one CTA per SM (two sharing an SM, as they do when they take
    // SMs while the scorer's CTAs finish, were 40% slower)
    const size_t smem = std::max<size_t>((size_t)(kCandCap + kStageCap) * 8 + (size_t)per * 4, 120 * 1024);
    const int vec = T_len % 4 == 0 && reinterpret_cast<uintptr_t>(scores) % 16 == 0;
    if ((e = ensure_smem((const void*)k_topk_fused, smem)) != cudaSuccess) return e;
    e = launch_pdl(k_topk_fused, dim3(kTopkCluster, H_kv), dim3(kTopkThreads), smem, st, scores, T_len, B_e, sel, per,
                   hist, vec, cosine_bins ? 1 : 0);
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
