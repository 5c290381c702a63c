// Query subselection: mean query, cosine to it, keep the N_q least similar.
// Method: QUOKA paper summary, "Query Subselection"; QUOKA Explained, "Pick
// the queries that disagree with the crowd".
//
// Three small launches (the stage reads Q about twice, ~2 x 17 MB at a
// 32-head 2048-token chunk, and is not on the critical byte path):
//   k_qstats : per (head, 64-row block) row norms |q| and partial column sums
//   k_qcos   : per (head, 64-row block) M_q from the partials (fixed order,
//              deterministic), then cos(q, M_q) for the block's rows
//   k_qselect: per selection row (query head, or KV group with the cosine
//              averaged over the group's heads) a shared-memory bitonic sort of
//              (key(cos), position) pairs; the first N_q are re-sorted by position.
#include "common.cuh"
#include "launch.h"

namespace quoka {

constexpr int kRowsPerBlock = 64;

template <typename T, int D>
__global__ void __launch_bounds__(256) k_qstats(const T* __restrict__ Q, int C, float* __restrict__ qnorm,
                                                float* __restrict__ qpart) {
  constexpr int E = D / 32;
  const int h = blockIdx.y, blk = blockIdx.x, nblk = gridDim.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float part[E];
#pragma unroll
  for (int j = 0; j < E; ++j) part[j] = 0.f;
  for (int r = warp; r < kRowsPerBlock; r += 8) {
    const int c = blk * kRowsPerBlock + r;
    if (c >= C) break;
    const T* q = Q + ((size_t)h * C + c) * D;
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < E; ++j) {
      float x = to_f32(q[lane + 32 * j]);
      part[j] += x;
      ss = fmaf(x, x, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) qnorm[(size_t)h * C + c] = sqrtf(ss);
  }
  __shared__ float sp[8][D];
#pragma unroll
  for (int j = 0; j < E; ++j) sp[warp][lane + 32 * j] = part[j];
  __syncthreads();
  if (threadIdx.x < D) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += sp[w][threadIdx.x];
    qpart[((size_t)h * nblk + blk) * D + threadIdx.x] = s;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(256) k_qcos(const T* __restrict__ Q, int C, const float* __restrict__ qpart,
                                              const float* __restrict__ qnorm, float* __restrict__ qcos) {
  constexpr int E = D / 32;
  const int h = blockIdx.y, blk = blockIdx.x, nblk = gridDim.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ float M[D];
  __shared__ float mnorm;
  if (threadIdx.x < D) {
    float s = 0.f;
    for (int b = 0; b < nblk; ++b) s += qpart[((size_t)h * nblk + b) * D + threadIdx.x];
    M[threadIdx.x] = s / (float)C;
  }
  __syncthreads();
  if (warp == 0) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < E; ++j) ss = fmaf(M[lane + 32 * j], M[lane + 32 * j], ss);
    ss = warp_sum(ss);
    if (lane == 0) mnorm = fmaxf(sqrtf(ss), kNormEps);
  }
  __syncthreads();
  for (int r = warp; r < kRowsPerBlock; r += 8) {
    const int c = blk * kRowsPerBlock + r;
    if (c >= C) break;
    const T* q = Q + ((size_t)h * C + c) * D;
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < E; ++j) dot = fmaf(to_f32(q[lane + 32 * j]), M[lane + 32 * j], dot);
    dot = warp_sum(dot);
    if (lane == 0) qcos[(size_t)h * C + c] = dot / (fmaxf(qnorm[(size_t)h * C + c], kNormEps) * mnorm);
  }
}

// Ascending bitonic sort of n (a power of two) 64-bit keys in shared memory.
__device__ void bitonic_sort_u64(uint64_t* a, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const bool up = (i & k) == 0;
          const uint64_t x = a[i], y = a[ixj];
          if ((x > y) == up) {
            a[i] = y;
            a[ixj] = x;
          }
        }
      }
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(1024) k_qselect(const float* __restrict__ qcos, int C, int G_avg, int n_sel,
                                                  int npow2, int32_t* __restrict__ q_idx) {
  extern __shared__ uint64_t keys[];
  const int row = blockIdx.x;
  for (int c = threadIdx.x; c < npow2; c += blockDim.x) {
    uint64_t key = ~0ull;
    if (c < C) {
      float u;
      if (G_avg == 1) {
        u = qcos[(size_t)row * C + c];
      } else {
        float s = 0.f;
        for (int k = 0; k < G_avg; ++k) s += qcos[((size_t)row * G_avg + k) * C + c];
        u = s / (float)G_avg;
      }
      key = ((uint64_t)order_key(u) << 32) | (uint32_t)c;   // smallest cosine first, then lowest position
    }
    keys[c] = key;
  }
  __syncthreads();
  bitonic_sort_u64(keys, npow2);
  for (int i = threadIdx.x; i < npow2; i += blockDim.x) keys[i] = (i < n_sel) ? (keys[i] & 0xffffffffull) : ~0ull;
  __syncthreads();
  bitonic_sort_u64(keys, npow2);
  for (int i = threadIdx.x; i < n_sel; i += blockDim.x) q_idx[(size_t)row * n_sel + i] = (int32_t)keys[i];
}

template <typename T, int D>
static cudaError_t qsel_impl(const void* Q, int H_q, int G_avg, int C, int n_sel, int32_t* q_idx,
                             float* qnorm, float* qpart, float* qcos, cudaStream_t st) {
  const int nblk = (C + kRowsPerBlock - 1) / kRowsPerBlock;
  dim3 grid(nblk, H_q);
  k_qstats<T, D><<<grid, 256, 0, st>>>((const T*)Q, C, qnorm, qpart);
  k_qcos<T, D><<<grid, 256, 0, st>>>((const T*)Q, C, qpart, qnorm, qcos);
  int npow2 = 32;
  while (npow2 < C) npow2 <<= 1;
  const size_t smem = (size_t)npow2 * sizeof(uint64_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_qselect, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int rows = H_q / G_avg;
  k_qselect<<<rows, 1024, smem, st>>>(qcos, C, G_avg, n_sel, npow2, q_idx);
  count_launches(3);
  return cudaGetLastError();
}

cudaError_t launch_select_queries(int dtype, int d, const void* Q, int H_q, int G_avg, int C, int n_sel,
                                  int32_t* q_idx, float* qnorm, float* qpart, float* qcos, cudaStream_t st) {
  if (dtype == 0) {
    return d == 64 ? qsel_impl<__nv_bfloat16, 64>(Q, H_q, G_avg, C, n_sel, q_idx, qnorm, qpart, qcos, st)
                   : qsel_impl<__nv_bfloat16, 128>(Q, H_q, G_avg, C, n_sel, q_idx, qnorm, qpart, qcos, st);
  }
  return d == 64 ? qsel_impl<float, 64>(Q, H_q, G_avg, C, n_sel, q_idx, qnorm, qpart, qcos, st)
                 : qsel_impl<float, 128>(Q, H_q, G_avg, C, n_sel, q_idx, qnorm, qpart, qcos, st);
}

}  // namespace quoka
