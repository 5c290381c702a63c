// Top-B history keys per KV head (QUOKA Explained, "From scores to a smaller
// KV set"; QUOKA paper summary, "Chunked Prefill with QUOKA").
//
// One CTA per KV head.  Scores are mapped to order-preserving 32-bit keys and
// an MSB-first radix select (4 digits of 8 bits, shared-memory histograms)
// finds the exact B-th largest key theta and how many keys equal to theta
// still have to be taken.  A final pass in position order writes every key
// above theta plus the lowest-position keys equal to theta, so the output is
// ascending and ties go to the lower position.
#include "common.cuh"
#include "launch.h"

namespace quoka {

constexpr int kTopkThreads = 1024;

__global__ void __launch_bounds__(kTopkThreads) k_topk_radix(const float* __restrict__ scores, int T_len, int B_e,
                                                             int32_t* __restrict__ sel) {
  const int g = blockIdx.x;
  const float* s = scores + (size_t)g * T_len;
  int32_t* out = sel + (size_t)g * B_e;
  __shared__ unsigned int hist[256];
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int s_need;
  __shared__ int scan_scratch[32];
  if (threadIdx.x == 0) {
    s_prefix = 0;
    s_mask = 0;
    s_need = B_e;
  }
  __syncthreads();
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (threadIdx.x < 256) hist[threadIdx.x] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix, mask = s_mask;
    for (int t = threadIdx.x; t < T_len; t += blockDim.x) {
      const uint32_t k = order_key(s[t]);
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int need = s_need, cum = 0, b = 255;
      for (; b > 0; --b) {
        if (cum + (int)hist[b] >= need) break;
        cum += (int)hist[b];
      }
      s_need = need - cum;
      s_prefix = prefix | ((uint32_t)b << shift);
      s_mask = mask | (255u << shift);
    }
    __syncthreads();
  }
  const uint32_t theta = s_prefix;
  const int r = s_need;   // keys equal to theta still to take, lowest positions first
  // Position-ordered compaction over contiguous per-thread ranges.
  const int per = (T_len + blockDim.x - 1) / blockDim.x;
  const int t0 = min(T_len, (int)threadIdx.x * per), t1 = min(T_len, t0 + per);
  int n_gt = 0, n_eq = 0;
  for (int t = t0; t < t1; ++t) {
    const uint32_t k = order_key(s[t]);
    n_gt += k > theta;
    n_eq += k == theta;
  }
  int total;
  const int eq_base = block_exclusive_scan(n_eq, scan_scratch, &total);
  const int take_eq = max(0, min(n_eq, r - eq_base));
  const int out_base = block_exclusive_scan(n_gt + take_eq, scan_scratch, &total);
  int o = out_base, eq_seen = 0;
  for (int t = t0; t < t1 && o < B_e; ++t) {     // o < B_e always holds; the test only guards the store
    const uint32_t k = order_key(s[t]);
    if (k > theta) {
      out[o++] = t;
    } else if (k == theta) {
      if (eq_seen < take_eq) out[o++] = t;
      ++eq_seen;
    }
  }
}

__global__ void k_iota_rows(int32_t* __restrict__ sel, int rows, int n) {
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
    k_iota_rows<<<blocks, 256, 0, st>>>(sel, H_kv, T_len);
    count_launches(1);
    return cudaGetLastError();
  }
  k_topk_radix<<<H_kv, kTopkThreads, 0, st>>>(scores, T_len, B_e, sel);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace quoka
