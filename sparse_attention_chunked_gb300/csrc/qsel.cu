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
//              averaged over the group's heads) an exact block radix select of
//              the N_q smallest cosines (keys = inverted order-mapped cosines,
//              so ties go to the lower position), written in position order.
#include "common.cuh"
#include "launch.h"
#include "radix_select.cuh"

namespace quoka {

constexpr int kRowsPerBlock = 64;
constexpr int kRowsPerWarp = kRowsPerBlock / 8;

// E consecutive elements of a row per lane, loaded as one vector.
template <typename T, int E>
struct alignas(sizeof(T) * E) RowSlice {
  T v[E];
};

// Loads the warp's kRowsPerWarp rows (lane holds elements lane*E .. lane*E+E-1),
// all loads issued before any use; rows at or beyond C read as zero.
template <typename T, int D>
__device__ __forceinline__ void load_rows(const T* __restrict__ Q, int h, int C, int c0, float (*x)[D / 32]) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  RowSlice<T, E> raw[kRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int c = c0 + r;
    if (c < C) raw[r] = *reinterpret_cast<const RowSlice<T, E>*>(Q + ((size_t)h * C + c) * D + lane * E);
  }
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
    for (int j = 0; j < E; ++j) x[r][j] = (c0 + r < C) ? to_f32(raw[r].v[j]) : 0.f;
}

template <typename T, int D>
__global__ void __launch_bounds__(256) k_qstats(const T* __restrict__ Q, int C, float* __restrict__ qnorm,
                                                float* __restrict__ qpart) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int E = D / 32;
  const int h = blockIdx.y, blk = blockIdx.x, nblk = gridDim.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = blk * kRowsPerBlock + warp * kRowsPerWarp;
  float x[kRowsPerWarp][E];
  load_rows<T, D>(Q, h, C, c0, x);
  float part[E], ss[kRowsPerWarp];
#pragma unroll
  for (int j = 0; j < E; ++j) part[j] = 0.f;
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    ss[r] = 0.f;
#pragma unroll
    for (int j = 0; j < E; ++j) {
      part[j] += x[r][j];
      ss[r] = fmaf(x[r][j], x[r][j], ss[r]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) ss[r] += __shfl_xor_sync(0xffffffffu, ss[r], o);
  if (lane < kRowsPerWarp) {
    float v = ss[0];
#pragma unroll
    for (int r = 1; r < kRowsPerWarp; ++r) v = lane == r ? ss[r] : v;
    if (c0 + lane < C) qnorm[(size_t)h * C + c0 + lane] = sqrtf(v);
  }
  __shared__ float sp[8][D];
#pragma unroll
  for (int j = 0; j < E; ++j) sp[warp][lane * E + j] = part[j];
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
  pdl_launch_dependents();
  pdl_wait();
  constexpr int E = D / 32;
  const int h = blockIdx.y, blk = blockIdx.x, nblk = gridDim.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = blk * kRowsPerBlock + warp * kRowsPerWarp;
  float x[kRowsPerWarp][E];
  load_rows<T, D>(Q, h, C, c0, x);                 // issued before the mean is ready
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
  float m[E];
#pragma unroll
  for (int j = 0; j < E; ++j) m[j] = M[lane * E + j];
  float dot[kRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    dot[r] = 0.f;
#pragma unroll
    for (int j = 0; j < E; ++j) dot[r] = fmaf(x[r][j], m[j], dot[r]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) dot[r] += __shfl_xor_sync(0xffffffffu, dot[r], o);
  if (lane < kRowsPerWarp && c0 + lane < C) {
    float v = dot[0];
#pragma unroll
    for (int r = 1; r < kRowsPerWarp; ++r) v = lane == r ? dot[r] : v;
    const int c = c0 + lane;
    qcos[(size_t)h * C + c] = v / (fmaxf(qnorm[(size_t)h * C + c], kNormEps) * mnorm);
  }
}

__global__ void __launch_bounds__(256) k_qselect(const float* __restrict__ qcos, int C, int G_avg, int n_sel,
                                                  int32_t* __restrict__ q_idx) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ __align__(16) uint32_t keys_s[];
  __shared__ RadixSelectShared rs;
  const int row = blockIdx.x;
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    float u;
    if (G_avg == 1) {
      u = qcos[(size_t)row * C + c];
    } else {
      float s = 0.f;
      for (int k = 0; k < G_avg; ++k) s += qcos[((size_t)row * G_avg + k) * C + c];
      u = s / (float)G_avg;
    }
    keys_s[c] = ~order_key(u);   // the largest key is the smallest cosine
  }
  __syncthreads();
  block_radix_topk4(reinterpret_cast<const uint4*>(keys_s), C, n_sel, q_idx + (size_t)row * n_sel, rs);
}

template <typename T, int D>
static cudaError_t qsel_impl(const void* Q, int H_q, int G_avg, int C, int n_sel, int32_t* q_idx,
                             float* qnorm, float* qpart, float* qcos, cudaStream_t st) {
  const int nblk = (C + kRowsPerBlock - 1) / kRowsPerBlock;
  dim3 grid(nblk, H_q);
  cudaError_t e = launch_pdl(k_qstats<T, D>, grid, dim3(256), 0, st, (const T*)Q, C, qnorm, qpart);
  if (e != cudaSuccess) return e;
  e = launch_pdl(k_qcos<T, D>, grid, dim3(256), 0, st, (const T*)Q, C, (const float*)qpart, (const float*)qnorm, qcos);
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)((C + 3) & ~3) * sizeof(uint32_t);   // C <= 8192: at most 32 KB
  const int rows = H_q / G_avg;
  e = launch_pdl(k_qselect, dim3(rows), dim3(256), smem, st, (const float*)qcos, C, G_avg, n_sel, q_idx);
  if (e != cudaSuccess) return e;
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
