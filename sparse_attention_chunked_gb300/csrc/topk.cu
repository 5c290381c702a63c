// Top-B history keys per KV head (QUOKA Explained, "From scores to a smaller
// KV set"; QUOKA paper summary, "Chunked Prefill with QUOKA").
//
// One CTA (1024 threads) per KV head runs an exact block radix select
// (radix_select.cuh) on the order-preserving 32-bit keys of the scores; when
// the head's keys fit in shared memory (T <= 48K) they are loaded once and all
// passes run from shared memory, otherwise every pass re-reads the scores
// from global memory (they are L2-resident right after the scoring kernel).
// The output is ascending and ties go to the lower position.
#include "common.cuh"
#include "launch.h"
#include "radix_select.cuh"

namespace quoka {

constexpr int kTopkThreads = 1024;
constexpr int kTopkSmemKeys = 48 * 1024;   // keys cached in shared memory (192 KB)

__global__ void __launch_bounds__(kTopkThreads) k_topk_radix(const float* __restrict__ scores, int T_len, int B_e,
                                                             int32_t* __restrict__ sel, int cache) {
  extern __shared__ uint32_t keys_s[];
  __shared__ RadixSelectShared rs;
  const int g = blockIdx.x;
  const float* s = scores + (size_t)g * T_len;
  int32_t* out = sel + (size_t)g * B_e;
  if (cache) {
    for (int i = threadIdx.x; i < T_len; i += blockDim.x) keys_s[i] = order_key(s[i]);
    __syncthreads();
    block_radix_topk([&](int i) { return keys_s[i]; }, T_len, B_e, out, rs);
  } else {
    block_radix_topk([&](int i) { return order_key(s[i]); }, T_len, B_e, out, rs);
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
  const int cache = T_len <= kTopkSmemKeys ? 1 : 0;
  const size_t smem = cache ? (size_t)T_len * 4 : 0;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_topk_radix, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  k_topk_radix<<<H_kv, kTopkThreads, smem, st>>>(scores, T_len, B_e, sel, cache);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace quoka
