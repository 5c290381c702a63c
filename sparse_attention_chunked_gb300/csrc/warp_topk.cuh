// Warp-level bitonic networks over L = 32 * P 64-bit elements, element
// e = p * 32 + lane held in register v[p] of lane `lane`.  Used for small
// top-k selections (query subselection keeps N_q of a chunk's positions),
// where a comparison network finishes in a few hundred cycles while a radix
// select is bound by its barriers.
//
// Elements are composite keys (key << 32) | (0xFFFFFFFF - position): larger
// composite = larger key, or the same key at a lower position, so "the L
// largest composites" is the exact top-L with ties to the lower position.
// 0 is smaller than every composite and pads short lists.
#pragma once

#include <stdint.h>

namespace quoka {

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t x, int m) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)x, m);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(x >> 32), m);
  return ((uint64_t)hi << 32) | lo;
}

__device__ __forceinline__ uint64_t shfl_u64(uint64_t x, int src) {
  const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)x, src);
  const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(x >> 32), src);
  return ((uint64_t)hi << 32) | lo;
}

// One compare-exchange step of distance j inside bitonic blocks of size k:
// within each block the larger element goes to the lower index when
// `desc_block` says so for that block, else to the higher index.
template <int P, bool kAllDescending>
__device__ __forceinline__ void bitonic_step(uint64_t (&v)[P], int k, int j) {
  const int lane = threadIdx.x & 31;
  if (j >= 32) {
    const int pj = j >> 5;
#pragma unroll
    for (int p = 0; p < P; ++p) {
      const int q = p ^ pj;
      if (q > p) {
        const int e = p * 32 + lane;
        const bool desc = kAllDescending || (e & k) == 0;
        const uint64_t a = v[p], b = v[q];
        const bool swap = desc ? (a < b) : (a > b);
        v[p] = swap ? b : a;
        v[q] = swap ? a : b;
      }
    }
  } else {
#pragma unroll
    for (int p = 0; p < P; ++p) {
      const int e = p * 32 + lane;
      const uint64_t o = shfl_xor_u64(v[p], j);
      const bool lower = (lane & j) == 0;
      const bool desc = kAllDescending || (e & k) == 0;
      // lower index keeps the larger (desc) or the smaller (asc) of the pair
      const bool keep_max = desc == lower;
      v[p] = keep_max ? (v[p] > o ? v[p] : o) : (v[p] < o ? v[p] : o);
    }
  }
}

// Sort the warp's L elements in descending order.
template <int P>
__device__ __forceinline__ void warp_sort_desc(uint64_t (&v)[P]) {
  constexpr int L = 32 * P;
#pragma unroll
  for (int k = 2; k <= L; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) bitonic_step<P, false>(v, k, j);
}

// a, b sorted descending; afterwards a holds the L largest of a and b, sorted descending.
template <int P>
__device__ __forceinline__ void warp_merge_desc(uint64_t (&a)[P], const uint64_t (&b)[P]) {
  constexpr int L = 32 * P;
  const int lane = threadIdx.x & 31;
  // a[i] vs b[L - 1 - i]: the larger of each pair forms a bitonic sequence holding the top L
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const uint64_t br = shfl_u64(b[P - 1 - p], 31 - lane);
    a[p] = a[p] > br ? a[p] : br;
  }
#pragma unroll
  for (int j = L >> 1; j > 0; j >>= 1) bitonic_step<P, true>(a, L, j);
}

}  // namespace quoka
