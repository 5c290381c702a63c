// Row gather of the selected history keys/values (QUOKA Explained, "From
// scores to a smaller KV set": the value comes with its key) and the cache
// append of a processed chunk (QUOKA Explained, "MEAN and MAX do different
// jobs": nothing is evicted).  Both are 16-byte vector copies, one vector per
// thread, grid-stride.
#include "common.cuh"
#include "launch.h"

namespace quoka {

// K_sel[g, j] = K_hist[g, sel[g, j]] and likewise V; row = vec_per_row uint4.
// A thread copies the same 16 bytes of the key row and of the value row, so
// the index is read once for both and the two loads are in flight together.
// An index outside [0, T_len) is never dereferenced: its row is written as
// zeros and QUOKA_ERR_DEVICE is recorded in hdr (when given) with the row.
__global__ void k_gather_rows(const uint4* __restrict__ K, const uint4* __restrict__ V, int64_t head_stride_vec,
                              const int32_t* __restrict__ sel, int H_kv, int B_e, int vec_per_row, int T_len,
                              uint4* __restrict__ Ks, uint4* __restrict__ Vs, WsHeader* hdr) {
  pdl_launch_dependents();   // early: the attention's prologue overlaps this copy
  pdl_wait_for(K, V, sel);
  const size_t per_mat = (size_t)H_kv * B_e * vec_per_row;
  for (size_t w = blockIdx.x * (size_t)blockDim.x + threadIdx.x; w < per_mat; w += (size_t)gridDim.x * blockDim.x) {
    const int v = (int)(w % vec_per_row);
    const size_t row = w / vec_per_row;              // g * B_e + j
    const int g = (int)(row / B_e);
    const int t = sel[row];
    if ((unsigned)t >= (unsigned)T_len) {
      if (v == 0) record_error(hdr, 7u /* QUOKA_ERR_DEVICE */, (unsigned)row);
      Ks[w] = Vs[w] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    const size_t off = (size_t)g * head_stride_vec + (size_t)t * vec_per_row + v;
    const uint4 k = K[off], x = V[off];
    Ks[w] = k;
    Vs[w] = x;
  }
}

// K_hist[g, T + c] = K_chunk[g, c] and likewise V.
__global__ void k_append_rows(uint4* __restrict__ K, uint4* __restrict__ V, int64_t head_stride_vec, int T_len,
                              const uint4* __restrict__ Kc, const uint4* __restrict__ Vc, int H_kv, int C,
                              int vec_per_row) {
  pdl_wait_for(Kc, Vc);
  const size_t per_mat = (size_t)H_kv * C * vec_per_row;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < 2 * per_mat;
       i += (size_t)gridDim.x * blockDim.x) {
    const bool is_v = i >= per_mat;
    const size_t w = is_v ? i - per_mat : i;
    const int v = (int)(w % vec_per_row);
    const size_t row = w / vec_per_row;              // g * C + c
    const int g = (int)(row / C), c = (int)(row % C);
    uint4* dst = (is_v ? V : K) + (size_t)g * head_stride_vec + (size_t)(T_len + c) * vec_per_row + v;
    *dst = (is_v ? Vc : Kc)[w];
  }
  pdl_launch_dependents();   // dependents launch once this CTA is done
}

// Key-norm cache: inv[g * inv_stride + t] = 1 / max(|K[g, t]|, eps) for
// t in [t0, t1).  One warp per key row; the squared norm is summed in fp32
// over the row's bf16 or fp32 elements.
template <typename T, int D>
__global__ void __launch_bounds__(256) k_key_inv_norms(const T* __restrict__ K, int64_t head_stride, int t0, int t1,
                                                       int H_kv, float* __restrict__ inv, int64_t inv_stride) {
  pdl_wait_for(K);
  constexpr int E = D / 32;
  const int n = t1 - t0;
  const size_t rows = (size_t)H_kv * n;
  const int lane = threadIdx.x & 31;
  for (size_t w = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5; w < rows;
       w += ((size_t)gridDim.x * blockDim.x) >> 5) {
    const int g = (int)(w / n), t = t0 + (int)(w % n);
    const T* k = K + (size_t)g * head_stride + (size_t)t * D;
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const float x = to_f32(k[lane + 32 * j]);
      ss = fmaf(x, x, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) inv[(size_t)g * inv_stride + t] = 1.0f / fmaxf(sqrtf(ss), kNormEps);
  }
  pdl_launch_dependents();   // dependents launch once this CTA is done
}

static int grid_for(size_t work) {
  size_t b = (work + 255) / 256;
  return (int)(b < 152 * 16 ? (b == 0 ? 1 : b) : 152 * 16);
}

cudaError_t launch_gather(int elt_bytes, int d, const void* K, const void* V, int64_t head_stride, const int32_t* sel,
                          int H_kv, int B_e, int T_len, void* Ks, void* Vs, WsHeader* hdr, cudaStream_t st) {
  if (B_e == 0) return cudaSuccess;
  const int vpr = d * elt_bytes / 16;
  const int64_t hsv = head_stride * elt_bytes / 16;
  cudaError_t e = launch_pdl(k_gather_rows, dim3(grid_for((size_t)H_kv * B_e * vpr)), dim3(256), 0, st,
                             (const uint4*)K, (const uint4*)V, hsv, sel, H_kv, B_e, vpr, T_len, (uint4*)Ks, (uint4*)Vs,
                             hdr);
  count_launches(1);
  return e;
}

cudaError_t launch_append(int elt_bytes, int d, void* K, void* V, int64_t head_stride, int T_len, const void* Kc,
                          const void* Vc, int H_kv, int C, cudaStream_t st) {
  const int vpr = d * elt_bytes / 16;
  const int64_t hsv = head_stride * elt_bytes / 16;
  cudaError_t e = launch_pdl(k_append_rows, dim3(grid_for((size_t)2 * H_kv * C * vpr)), dim3(256), 0, st, (uint4*)K,
                             (uint4*)V, hsv, T_len, (const uint4*)Kc, (const uint4*)Vc, H_kv, C, vpr);
  count_launches(1);
  return e;
}

cudaError_t launch_key_inv_norms(int dtype, int d, const void* K, int64_t head_stride, int H_kv, int t0, int t1,
                                 float* inv, int64_t inv_stride, cudaStream_t st) {
  if (t1 <= t0) return cudaSuccess;
  const dim3 grid(grid_for((size_t)H_kv * (t1 - t0) * 32));
  cudaError_t e;
  if (dtype == 0) {
    if (d == 64)
      e = launch_pdl(k_key_inv_norms<__nv_bfloat16, 64>, grid, dim3(256), 0, st, (const __nv_bfloat16*)K, head_stride,
                     t0, t1, H_kv, inv, inv_stride);
    else
      e = launch_pdl(k_key_inv_norms<__nv_bfloat16, 128>, grid, dim3(256), 0, st, (const __nv_bfloat16*)K,
                     head_stride, t0, t1, H_kv, inv, inv_stride);
  } else {
    if (d == 64)
      e = launch_pdl(k_key_inv_norms<float, 64>, grid, dim3(256), 0, st, (const float*)K, head_stride, t0, t1, H_kv,
                     inv, inv_stride);
    else
      e = launch_pdl(k_key_inv_norms<float, 128>, grid, dim3(256), 0, st, (const float*)K, head_stride, t0, t1, H_kv,
                     inv, inv_stride);
  }
  count_launches(1);
  return e;
}

}  // namespace quoka
