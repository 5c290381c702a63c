// CUDA-core flash attention over [history rows ; causal chunk].
// Method: QUOKA paper summary, "Transformers and Attention" (softmax
// attention with a causal mask), "Chunked prefill" (the chunk attends to the
// earlier keys plus itself, causally), "QUOKA Method" (the reduced key set is
// fed to a dense attention kernel).
//
// This is the fp32 path (no TF32: every product and sum is an fp32 FMA) and
// the portable bf16 path.  A CTA owns 32 query rows of one head; each of its
// 4 warps owns 8 rows.  Keys stream through shared memory 32 at a time: lane
// j scores key j against a row, the warp does the online-softmax update with
// shuffles, and each lane accumulates d/32 output columns.
#include "common.cuh"
#include "launch.h"

namespace quoka {

constexpr int kAttRows = 32;   // query rows per CTA
constexpr int kAttKeys = 32;   // keys per shared-memory tile

template <typename T, int D>
__global__ void __launch_bounds__(128) k_attend_simt(const T* __restrict__ Q, const T* __restrict__ Kh,
                                                     const T* __restrict__ Vh, int64_t h_stride, int n_hist,
                                                     const T* __restrict__ Kc, const T* __restrict__ Vc, int C,
                                                     int G, float scale_log2, T* __restrict__ O,
                                                     float* __restrict__ lse) {
  pdl_wait_for(Q, Kh, Vh, Kc, Vc);
  constexpr int E = D / 32;
  constexpr int RPW = kAttRows / 4;   // rows per warp
  extern __shared__ float smem[];
  float* Qs = smem;                               // [32][D]
  float* Ks = Qs + kAttRows * D;                  // [32][D+1]
  float* Vs = Ks + kAttKeys * (D + 1);            // [32][D]
  const int h = blockIdx.y, g = h / G;
  const int q0 = blockIdx.x * kAttRows;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  for (int i = threadIdx.x; i < kAttRows * D; i += blockDim.x) {
    const int r = i / D, e = i % D;
    const int c = q0 + r;
    Qs[i] = c < C ? to_f32(Q[((size_t)h * C + c) * D + e]) : 0.f;
  }
  float m[RPW], l[RPW], acc[RPW][E];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[i][e] = 0.f;
  }
  const int last_row = min(C, q0 + kAttRows) - 1;
  const int n_keys = n_hist + last_row + 1;       // chunk keys beyond the last row are never seen
  for (int j0 = 0; j0 < n_keys; j0 += kAttKeys) {
    __syncthreads();
    for (int i = threadIdx.x; i < kAttKeys * D; i += blockDim.x) {
      const int jj = i / D, e = i % D;
      const int j = j0 + jj;
      float kv = 0.f, vv = 0.f;
      if (j < n_hist) {
        const size_t off = (size_t)g * h_stride + (size_t)j * D + e;
        kv = to_f32(Kh[off]);
        vv = to_f32(Vh[off]);
      } else if (j < n_keys) {
        const size_t off = ((size_t)g * C + (j - n_hist)) * D + e;
        kv = to_f32(Kc[off]);
        vv = to_f32(Vc[off]);
      }
      Ks[jj * (D + 1) + e] = kv;
      Vs[jj * D + e] = vv;
    }
    __syncthreads();
    const int j = j0 + lane;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const int r = warp * RPW + i;
      const int c = q0 + r;
      const bool valid = j < n_hist || (j < n_keys && (j - n_hist) <= c);
      float dot = 0.f;
#pragma unroll 16
      for (int e = 0; e < D; ++e) dot = fmaf(Qs[r * D + e], Ks[lane * (D + 1) + e], dot);
      const float x = valid ? dot * scale_log2 : -INFINITY;
      const float m_new = fmaxf(m[i], warp_max(x));
      if (m_new == -INFINITY) continue;            // nothing visible yet for this row (warp-uniform)
      const float p = exp2f(x - m_new);
      const float corr = exp2f(m[i] - m_new);
      l[i] = l[i] * corr + warp_sum(p);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[i][e] *= corr;
#pragma unroll 8
      for (int jj = 0; jj < kAttKeys; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[i][e] = fmaf(pj, Vs[jj * D + lane + 32 * e], acc[i][e]);
      }
      m[i] = m_new;
    }
  }
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const int c = q0 + warp * RPW + i;
    if (c >= C) continue;
    const float inv = 1.0f / l[i];
#pragma unroll
    for (int e = 0; e < E; ++e) O[((size_t)h * C + c) * D + lane + 32 * e] = from_f32<T>(acc[i][e] * inv);
    if (lse != nullptr && lane == 0) lse[(size_t)h * C + c] = m[i] * 0.69314718055994531f + logf(l[i]);
  }
  pdl_launch_dependents();   // dependents launch once this CTA is done
}

template <typename T, int D>
static cudaError_t attend_impl(const void* Q, const void* Kh, const void* Vh, int64_t h_stride, int n_hist,
                               const void* Kc, const void* Vc, int H_q, int C, int G, float scale, void* O,
                               float* lse, cudaStream_t st) {
  const size_t smem = sizeof(float) * (kAttRows * D + kAttKeys * (D + 1) + kAttKeys * D);
  cudaError_t e = ensure_smem((const void*)k_attend_simt<T, D>, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((C + kAttRows - 1) / kAttRows, H_q);
  const float scale_log2 = scale * 1.4426950408889634f;
  e = launch_pdl(k_attend_simt<T, D>, grid, dim3(128), smem, st, (const T*)Q, (const T*)Kh, (const T*)Vh, h_stride,
                 n_hist, (const T*)Kc, (const T*)Vc, C, G, scale_log2, (T*)O, lse);
  count_launches(1);
  return e;
}

cudaError_t launch_attend_simt(int dtype, int d, const void* Q, const void* Kh, const void* Vh, int64_t h_stride,
                               int n_hist, const void* Kc, const void* Vc, int H_q, int C, int G, float scale,
                               void* O, float* lse, cudaStream_t st) {
  if (dtype == 0)
    return d == 64 ? attend_impl<__nv_bfloat16, 64>(Q, Kh, Vh, h_stride, n_hist, Kc, Vc, H_q, C, G, scale, O, lse, st)
                   : attend_impl<__nv_bfloat16, 128>(Q, Kh, Vh, h_stride, n_hist, Kc, Vc, H_q, C, G, scale, O, lse, st);
  return d == 64 ? attend_impl<float, 64>(Q, Kh, Vh, h_stride, n_hist, Kc, Vc, H_q, C, G, scale, O, lse, st)
                 : attend_impl<float, 128>(Q, Kh, Vh, h_stride, n_hist, Kc, Vc, H_q, C, G, scale, O, lse, st);
}

}  // namespace quoka
