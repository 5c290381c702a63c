// Query subselection: mean query, cosine to it, keep the N_q least similar.
// Method: QUOKA paper summary, "Query Subselection"; QUOKA Explained, "Pick
// the queries that disagree with the crowd".
//
// A selection row is a query head, or a KV group with the cosine averaged
// over the group's heads.  Its N_q smallest cosines are kept (keys =
// inverted order-mapped cosines, so ties go to the lower position), written
// in position order.
//
// k_qselect_fused: a cluster of CL CTAs per selection row (8; 4 when a
// quarter of the chunk fits one staging piece, so that short chunks do not
// spread thin over twice the CTAs), CTA r owning the r-th CL-th of the chunk
// positions.  Each CTA copies its slice of Q into
// shared memory with bulk copies (64-row chunks, each on its own mbarrier, so
// the arithmetic starts as the first chunk lands), takes the row norms |q|
// and the column sums; the cluster adds the slices' sums through distributed
// shared memory in rank order (deterministic) for M_q; each CTA then computes
// cos(q, M_q) for its rows from shared memory (a slice larger than the 64 KB
// staging buffer, or a group of several heads, is staged again piece by
// piece, from L2) into shared-memory keys.  For N_q <= 256 the selection is a
// bitonic network (warp_topk.cuh): each warp keeps the top L >= N_q of its
// keys, warp 0 merges its CTA's lists, CTA 0 merges the cluster's lists
// through distributed shared memory and writes the winners' positions in
// ascending order; larger N_q take the cluster radix select of
// cluster_topk.cuh.
//
// Mean pooling runs k_qselect_fused with one query head per cluster, writing
// each head's cosines to the workspace, then k_qselect_groups (one CTA per KV
// group) sums a group's cosines in head order and selects by a histogram: the two passes over Q then run
// on one cluster per query head instead of one per KV group (a group of four
// heads took four times as long on a quarter of the clusters).  Where the
// cosines have no room (the workspace-free entry point's fixed array), the
// fused kernel takes whole groups in one launch.
#include "common.cuh"
#include "launch.h"
#include <cooperative_groups.h>

#include "block_select.cuh"
#include "cluster_topk.cuh"
#include "tc_common.cuh"
#include "radix_select.cuh"
#include "warp_topk.cuh"

namespace cg = cooperative_groups;

namespace quoka {

constexpr int kRowsPerBlock = 64;
constexpr int kRowsPerWarp = kRowsPerBlock / 8;

// E consecutive elements of a row per lane, loaded as one vector.
template <typename T, int E>
struct alignas(sizeof(T) * E) RowSlice {
  T v[E];
};

constexpr int kSelCluster = 8;                      // the largest cluster
constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
static_assert(kSelWarps >= kSelCluster, "warp q of CTA 0 fetches the list of CTA q");
static_assert(kRowsPerWarp == 8, "the reduce-scatter below is written for 8 rows");

// Warp sums of 8 rows at once: v[r] is this lane's part of row r; afterwards
// every lane holds the full sum of row rs_row(lane) (lanes 4k .. 4k+3 share a
// row).  9 shuffles instead of 8 separate 5-step butterflies.
__device__ __forceinline__ int rs_row(int lane) { return ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1); }
__device__ __forceinline__ float reduce_scatter8(const float (&v)[8]) {
  const int lane = threadIdx.x & 31;
  const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0, b2 = (lane & 4) != 0;
  float a[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)   // keep rows 4*b4 .. 4*b4+3, send the partner the other four
    a[j] = (b4 ? v[j + 4] : v[j]) + __shfl_xor_sync(0xffffffffu, b4 ? v[j] : v[j + 4], 16);
  float b[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) b[j] = (b3 ? a[j + 2] : a[j]) + __shfl_xor_sync(0xffffffffu, b3 ? a[j] : a[j + 2], 8);
  float c = (b2 ? b[1] : b[0]) + __shfl_xor_sync(0xffffffffu, b2 ? b[0] : b[1], 4);
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  c += __shfl_xor_sync(0xffffffffu, c, 1);
  return c;
}

constexpr int kSelChunkRows = 64;                   // rows per bulk copy / mbarrier
constexpr size_t kSelStageBytes = 64 * 1024;          // shared-memory staging of Q rows
constexpr int kSelMaxChunks = 16;

// Rows of one staged piece of a slice (a multiple of kSelChunkRows).
__host__ __device__ inline int qselect_piece_rows(int D, int elt) {
  return (int)(kSelStageBytes / ((size_t)D * elt)) / kSelChunkRows * kSelChunkRows;
}
// Offset (in floats, after the staging buffer) of the selection lists in
// k_qselect_fused's dynamic shared memory, and the total size in bytes.
__host__ __device__ inline size_t qselect_lists_offset(int per, int G_avg, int D) {
  return ((size_t)per + (size_t)per + (size_t)G_avg * per + 2 * (size_t)G_avg * D + (size_t)G_avg + 1) & ~(size_t)1;
}
static size_t qselect_fused_smem(int per, int G_avg, int D, int sel_p) {
  return kSelStageBytes + qselect_lists_offset(per, G_avg, D) * sizeof(float) +
         (size_t)(kSelWarps + 1) * 32 * sel_p * sizeof(uint64_t);
}

// Top n_sel (<= 32 * P) of the row's keys, split over the cluster as in
// k_qselect_fused; out receives their positions in ascending order.  lists:
// (kSelWarps + 1) * 32 * P composites of shared memory.  The warps' lists are
// merged as a tree, then CTA 0's warps fetch the CTAs' lists (one each) and
// merge those as a tree.  Every CTA passes the same two cluster barriers; CTA
// 0 alone continues after the second.
template <int P, int CL>
__device__ void cluster_warp_topk(cg::cluster_group& cluster, const uint32_t* keys_s, int n, int t0, int n_sel,
                                  uint64_t* lists, int32_t* __restrict__ out) {
  constexpr int L = 32 * P;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t run[P];
#pragma unroll
  for (int p = 0; p < P; ++p) run[p] = 0ull;
  for (int seg = warp; seg * L < n; seg += kSelWarps) {
    uint64_t v[P];
#pragma unroll
    for (int p = 0; p < P; ++p) {
      const int i = seg * L + p * 32 + lane;
      v[p] = i < n ? (((uint64_t)keys_s[i] << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)(t0 + i))) : 0ull;
    }
    warp_sort_desc<P>(v);
    warp_merge_desc<P>(run, v);
  }
  // tree merge of the warps' lists: after it list 0 (and warp 0's run) is the CTA's top L
  auto tree_merge = [&]() {
#pragma unroll
    for (int p = 0; p < P; ++p) lists[warp * L + p * 32 + lane] = run[p];
    __syncthreads();
    for (int stride = 1; stride < kSelWarps; stride <<= 1) {
      if ((warp & (2 * stride - 1)) == 0) {
        uint64_t b[P];
#pragma unroll
        for (int p = 0; p < P; ++p) b[p] = lists[(warp + stride) * L + p * 32 + lane];
        warp_merge_desc<P>(run, b);
#pragma unroll
        for (int p = 0; p < P; ++p) lists[warp * L + p * 32 + lane] = run[p];
      }
      __syncthreads();
    }
  };
  tree_merge();
  // this CTA's list goes to the spare slot, where CTA 0 reads it
  if (warp == 0)
#pragma unroll
    for (int p = 0; p < P; ++p) lists[kSelWarps * L + p * 32 + lane] = run[p];
  cluster.sync();                                 // every CTA's list is ready
  const bool leader = cluster.block_rank() == 0;
  if (leader) {                                   // warp q of CTA 0 fetches CTA q's list (q < CL)
    if (warp < CL) {
      const uint64_t* rl = cluster.map_shared_rank(lists + kSelWarps * L, warp);
#pragma unroll
      for (int p = 0; p < P; ++p) run[p] = rl[p * 32 + lane];
    } else {
#pragma unroll
      for (int p = 0; p < P; ++p) run[p] = 0ull;
    }
  }
  cluster.sync();                                 // every remote read is done: the other CTAs may finish
  if (!leader) return;
  tree_merge();
  if (warp == 0) {
    // the first n_sel winners, by ascending position (0xFFFFFFFF - position, descending)
#pragma unroll
    for (int p = 0; p < P; ++p) run[p] = p * 32 + lane < n_sel ? (uint64_t)(uint32_t)run[p] : 0ull;
    warp_sort_desc<P>(run);
#pragma unroll
    for (int p = 0; p < P; ++p)
      if (p * 32 + lane < n_sel) out[p * 32 + lane] = (int32_t)(0xFFFFFFFFu - (uint32_t)run[p]);
  }
}

template <typename T, int D, int CL>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(kSelThreads, 2)
    k_qselect_fused(const T* __restrict__ Q, int C, int G_avg, int n_sel, int per, int sel_p,
                    int32_t* __restrict__ q_idx, float* __restrict__ cos_out, WsHeader* hdr) {
  constexpr int E = D / 32;
  extern __shared__ __align__(1024) uint8_t dsm_raw[];
  T* rows_s = reinterpret_cast<T*>(dsm_raw);                                 // staged rows of a piece
  float* dyn = reinterpret_cast<float*>(dsm_raw + kSelStageBytes);
  uint32_t* keys_s = reinterpret_cast<uint32_t*>(dyn);   // [per], per % 4 == 0
  float* u_s = dyn + per;                                // [per] cosine summed over the row's heads
  float* norm_s = u_s + per;                             // [G_avg][per]
  float* part_s = norm_s + (size_t)G_avg * per;          // [G_avg][D] column sums of this slice (read cluster-wide)
  float* mean_s = part_s + (size_t)G_avg * D;            // [G_avg][D]
  float* mnorm_s = mean_s + (size_t)G_avg * D;           // [G_avg]
  uint64_t* lists = reinterpret_cast<uint64_t*>(dyn + qselect_lists_offset(per, G_avg, D));
  __shared__ float sp[kSelWarps][D];
  __shared__ ClusterTopkShared tk;
  __shared__ uint64_t rbar[kSelMaxChunks];
  __shared__ int abort_flag;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.y;
  const int t0 = min(C, rank * per), n = min(C, t0 + per) - t0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int piece = qselect_piece_rows(D, (int)sizeof(T));
  const int npieces = (n + piece - 1) / piece;
  if (threadIdx.x == 0) {
    for (int c = 0; c < kSelMaxChunks; ++c) tc::mbar_init(&rbar[c], 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  for (int i = threadIdx.x; i < per; i += blockDim.x) u_s[i] = 0.f;
  __syncthreads();
  volatile int* abort = &abort_flag;
  pdl_wait_for(Q);   // Q may come from the previous kernel

  // Stage rows [p0, p0 + pn) of head k's slice; every thread calls it (it syncs), thread 0 issues.
  int round = 0;                                  // staging rounds so far: chunk barriers' phase
  int last_pn = 0;                                // rows of the last staged piece
  auto stage = [&](int k, int p0, int pn) {
    __syncthreads();                              // the previous piece is no longer read
    if (threadIdx.x == 0) {
      tc::fence_proxy_async_smem();               // generic reads of the buffer before the async writes
      const T* src = Q + ((size_t)(row * G_avg + k) * C + t0 + p0) * D;
      for (int c = 0; c * kSelChunkRows < pn; ++c) {
        const uint32_t bytes = (uint32_t)(min(kSelChunkRows, pn - c * kSelChunkRows) * D * (int)sizeof(T));
        tc::mbar_arrive_expect_tx(&rbar[c], bytes);
        tc::bulk_load(rows_s + (size_t)c * kSelChunkRows * D, src + (size_t)c * kSelChunkRows * D, bytes, &rbar[c]);
      }
    }
    ++round;
    last_pn = pn;
  };
  // the rows c0 .. c0+7 of the staged piece (pn rows), waiting for their chunk; false once a wait gave up
  auto rows_ready = [&](int c0) -> bool {
    bool ok = true;
    if (lane == 0) ok = tc::mbar_wait(&rbar[c0 / kSelChunkRows], (round - 1) & 1, abort, hdr, 0x301);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  };
  auto read_rows = [&](int c0, int pn, float (*x)[E]) {
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      RowSlice<T, E> raw;
      if (c0 + r < pn) raw = *reinterpret_cast<const RowSlice<T, E>*>(rows_s + (size_t)(c0 + r) * D + lane * E);
#pragma unroll
      for (int j = 0; j < E; ++j) x[r][j] = (c0 + r < pn) ? to_f32(raw.v[j]) : 0.f;
    }
  };

  // 1. row norms and column sums of this slice, head by head
  for (int k = 0; k < G_avg; ++k) {
    float part[E];
#pragma unroll
    for (int j = 0; j < E; ++j) part[j] = 0.f;
    for (int pi = 0; pi < npieces; ++pi) {
      const int p0 = pi * piece, pn = min(piece, n - p0);
      stage(k, p0, pn);
      for (int c0 = warp * kRowsPerWarp; c0 < pn; c0 += kSelWarps * kRowsPerWarp) {
        if (!rows_ready(c0)) break;
        float x[kRowsPerWarp][E];
        read_rows(c0, pn, x);
        float ss[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
          ss[r] = 0.f;
#pragma unroll
          for (int j = 0; j < E; ++j) {
            part[j] += x[r][j];
            ss[r] = fmaf(x[r][j], x[r][j], ss[r]);
          }
        }
        const float v = reduce_scatter8(ss);
        const int rr = rs_row(lane);
        if ((lane & 3) == 0 && c0 + rr < pn) norm_s[(size_t)k * per + p0 + c0 + rr] = sqrtf(v);
      }
    }
#pragma unroll
    for (int j = 0; j < E; ++j) sp[warp][lane * E + j] = part[j];
    __syncthreads();
    for (int t = threadIdx.x; t < D; t += blockDim.x) {
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kSelWarps; ++w) acc += sp[w][t];
      part_s[(size_t)k * D + t] = acc;
    }
    __syncthreads();
  }
  cluster.sync();

  // 2. M_q of every head of the row: the slices' sums in rank order, / C
  for (int i = threadIdx.x; i < G_avg * D; i += blockDim.x) {
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < CL; ++q) acc += cluster.map_shared_rank(part_s, q)[i];
    mean_s[i] = acc / (float)C;
  }
  __syncthreads();
  for (int k = warp; k < G_avg; k += kSelWarps) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < E; ++j) ss = fmaf(mean_s[k * D + lane + 32 * j], mean_s[k * D + lane + 32 * j], ss);
    ss = warp_sum(ss);
    if (lane == 0) mnorm_s[k] = fmaxf(sqrtf(ss), kNormEps);
  }
  __syncthreads();

  // 3. cos(q, M_q), summed over the row's heads in head order; the last staged
  //    piece is still in shared memory when the row has one head and one piece
  const bool resident = G_avg == 1 && npieces == 1;
  for (int k = 0; k < G_avg; ++k) {
    float m[E];
#pragma unroll
    for (int j = 0; j < E; ++j) m[j] = mean_s[k * D + lane * E + j];
    const float mn = mnorm_s[k];
    for (int pi = 0; pi < npieces; ++pi) {
      const int p0 = pi * piece, pn = min(piece, n - p0);
      if (!resident) stage(k, p0, pn);
      for (int c0 = warp * kRowsPerWarp; c0 < pn; c0 += kSelWarps * kRowsPerWarp) {
        if (!resident && !rows_ready(c0)) break;
        float x[kRowsPerWarp][E];
        read_rows(c0, pn, x);
        float dot[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
          dot[r] = 0.f;
#pragma unroll
          for (int j = 0; j < E; ++j) dot[r] = fmaf(x[r][j], m[j], dot[r]);
        }
        const float v = reduce_scatter8(dot);
        const int rr = rs_row(lane);
        if ((lane & 3) == 0 && c0 + rr < pn) {
          const int i = p0 + c0 + rr;
          u_s[i] += v / (fmaxf(norm_s[(size_t)k * per + i], kNormEps) * mn);
        }
      }
    }
  }
  __syncthreads();
  if (cos_out != nullptr) {   // one head per row: its cosines, for the group select (k_qselect_groups)
    for (int i = threadIdx.x; i < n; i += blockDim.x) cos_out[(size_t)row * C + t0 + i] = u_s[i];
  } else {
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const float v = G_avg > 1 ? u_s[i] / (float)G_avg : u_s[i];
      keys_s[i] = ~order_key(v);   // the largest key is the smallest cosine
    }
  }
  if (threadIdx.x == 0 && *abort && round > 0) {   // let the last staged copies land before the CTA can exit
    for (int c = 0; c * kSelChunkRows < last_pn; ++c) tc::mbar_drain(&rbar[c], (round - 1) & 1);
  }
  __syncthreads();
  if (cos_out != nullptr) {
    cluster.sync();   // keep part_s alive until every CTA has read it
    pdl_launch_dependents();
    return;
  }

  // 4. the n_sel least similar positions of the row
  int32_t* out = q_idx + (size_t)row * n_sel;
  if (n_sel >= C) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) out[t0 + i] = t0 + i;
    cluster.sync();   // keep part_s alive until every CTA has read it
    return;
  }
  switch (sel_p) {
    case 1: cluster_warp_topk<1, CL>(cluster, keys_s, n, t0, n_sel, lists, out); return;
    case 2: cluster_warp_topk<2, CL>(cluster, keys_s, n, t0, n_sel, lists, out); return;
    case 4: cluster_warp_topk<4, CL>(cluster, keys_s, n, t0, n_sel, lists, out); return;
    case 8: cluster_warp_topk<8, CL>(cluster, keys_s, n, t0, n_sel, lists, out); return;
    default: {
      auto key_at = [&](int i) -> uint32_t { return keys_s[i]; };
      cluster_radix_topk<CL>(cluster, true, reinterpret_cast<const uint4*>(keys_s), key_at, n, t0, n_sel, out,
                                      tk);
    }
  }
  pdl_launch_dependents();   // dependents launch once this CTA is done
}

// The group select of mean pooling: one CTA per KV group sums the cosines of
// the group's query heads (written by k_qselect_fused running one head per
// cluster) in head order and averages them, as the one-launch kernel does for
// a whole group, then keeps the n_sel least similar positions by the
// histogram select of block_select.cuh: the keys are inverted order keys of
// the averaged cosine, binned by the fixed-point bin of its negation (4096
// bins of width 1/2048 over [-1, 1], non-decreasing in the key).  Splitting
// the selection this way runs the heavy part (two passes over Q) on one
// cluster per query head instead of one per KV group.
constexpr int kRowSelThreads = 1024;

__global__ void __launch_bounds__(kRowSelThreads)
    k_qselect_groups(const float* __restrict__ qcos, int C, int G_avg, int n_sel, int32_t* __restrict__ q_idx) {
  extern __shared__ __align__(16) uint8_t rsel_raw[];
  uint2* cand = reinterpret_cast<uint2*>(rsel_raw);                // [C] (key, position)
  uint32_t* keys = reinterpret_cast<uint32_t*>(cand + C);          // [C]
  __shared__ BlockSelectShared bs;
  const int row = blockIdx.x;
  pdl_wait_for(qcos);
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    float u = 0.f;
    for (int k = 0; k < G_avg; ++k) u += qcos[((size_t)row * G_avg + k) * C + c];
    keys[c] = ~order_key(G_avg > 1 ? u / (float)G_avg : u);   // the largest key is the smallest cosine
  }
  __syncthreads();
  auto bin_of = [](uint32_t key) -> uint32_t { return score_bin(-key_float(~key), true); };
  block_select_top(keys, C, n_sel, q_idx + (size_t)row * n_sel, 0, cand, bs, bin_of);
  pdl_launch_dependents();   // dependents launch once this CTA is done
}

// CTAs per selection row: 4 when a quarter of the chunk fits one staging
// piece, else 8.
static int qselect_cluster(int d, int elt, int C) {
  return (C + 3) / 4 <= qselect_piece_rows(d, elt) ? 4 : kSelCluster;
}

// k_qselect_fused's parameters: slice length per CTA, list length
// 32 * sel_p >= n_sel (0: radix select), dynamic shared memory.
static void qselect_fused_plan(int d, int elt, int G_avg, int C, int n_sel, int* per, int* sel_p, size_t* smem) {
  const int cl = qselect_cluster(d, elt, C);
  *per = ((C + cl - 1) / cl + 3) & ~3;
  *sel_p = n_sel <= 32 ? 1 : n_sel <= 64 ? 2 : n_sel <= 128 ? 4 : n_sel <= 256 ? 8 : 0;
  *smem = qselect_fused_smem(*per, G_avg, d, *sel_p);
}

// The clustered kernel runs when its shared memory stays within 160 KB and Q
// is 16-byte aligned (bulk copies want 16-byte aligned rows).
static bool fused_fits(int d, int elt, const void* Q, int G_avg, int C, int n_sel) {
  int per, sel_p;
  size_t fsmem;
  qselect_fused_plan(d, elt, G_avg, C, n_sel, &per, &sel_p, &fsmem);
  return fsmem <= 160 * 1024 && ((uintptr_t)Q & 15u) == 0;
}

int select_queries_path(int dtype, int d, const void* Q, int H_q, int G_avg, int C, int n_sel, bool split_ok) {
  (void)H_q;
  const int elt = dtype == 0 ? 2 : 4;
  if (G_avg > 1 && split_ok && fused_fits(d, elt, Q, 1, C, n_sel)) return 2;
  if (fused_fits(d, elt, Q, G_avg, C, n_sel)) return 1;
  return 0;
}

template <typename T, int D, int CL>
static cudaError_t qsel_launch(dim3 grid, size_t smem, cudaStream_t st, const void* Q, int C, int G_run, int n_sel,
                               int per, int sel_p, int32_t* q_idx, float* cos_out, WsHeader* hdr) {
  cudaError_t e = ensure_smem((const void*)k_qselect_fused<T, D, CL>, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_qselect_fused<T, D, CL>, grid, dim3(kSelThreads), smem, st, (const T*)Q, C, G_run, n_sel, per,
                    sel_p, q_idx, cos_out, hdr);
}

template <typename T, int D>
static cudaError_t qsel_impl(const void* Q, int H_q, int G_avg, int C, int n_sel, int32_t* q_idx, float* qcos,
                             WsHeader* hdr, bool split_ok, cudaStream_t st) {
  const int rows = H_q / G_avg;
  const int path = select_queries_path(sizeof(T) == 2 ? 0 : 1, D, Q, H_q, G_avg, C, n_sel, split_ok);
  if (path == 0) return cudaErrorInvalidConfiguration;   // the callers check select_queries_path first
  const int G_run = path == 2 ? 1 : G_avg;   // the split runs one head per cluster
  int per, sel_p;
  size_t fsmem;
  qselect_fused_plan(D, (int)sizeof(T), G_run, C, n_sel, &per, &sel_p, &fsmem);
  const int cl = qselect_cluster(D, (int)sizeof(T), C);
  float* cos_out = path == 2 ? qcos : (float*)nullptr;
  const dim3 grid(cl, H_q / G_run);
  cudaError_t e = cl == 4 ? qsel_launch<T, D, 4>(grid, fsmem, st, Q, C, G_run, n_sel, per, sel_p, q_idx, cos_out, hdr)
                          : qsel_launch<T, D, kSelCluster>(grid, fsmem, st, Q, C, G_run, n_sel, per, sel_p, q_idx,
                                                           cos_out, hdr);
  count_launches(1);
  if (e != cudaSuccess || path == 1) return e;
  const size_t gsmem = (size_t)C * (sizeof(uint2) + sizeof(uint32_t));
  if ((e = ensure_smem((const void*)k_qselect_groups, gsmem)) != cudaSuccess) return e;
  e = launch_pdl(k_qselect_groups, dim3(rows), dim3(kRowSelThreads), gsmem, st, (const float*)qcos, C, G_avg, n_sel,
                 q_idx);
  count_launches(1);
  return e;
}

cudaError_t launch_select_queries(int dtype, int d, const void* Q, int H_q, int G_avg, int C, int n_sel,
                                  int32_t* q_idx, float* qcos, WsHeader* hdr, cudaStream_t st, bool split_ok) {
  if (dtype == 0) {
    return d == 64 ? qsel_impl<__nv_bfloat16, 64>(Q, H_q, G_avg, C, n_sel, q_idx, qcos, hdr, split_ok, st)
                   : qsel_impl<__nv_bfloat16, 128>(Q, H_q, G_avg, C, n_sel, q_idx, qcos, hdr, split_ok, st);
  }
  return d == 64 ? qsel_impl<float, 64>(Q, H_q, G_avg, C, n_sel, q_idx, qcos, hdr, split_ok, st)
                 : qsel_impl<float, 128>(Q, H_q, G_avg, C, n_sel, q_idx, qcos, hdr, split_ok, st);
}

}  // namespace quoka
