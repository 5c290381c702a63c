// Device helpers shared by the QUOKA kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace quoka {

constexpr float kNormEps = 1e-12f;   // norms below this are clamped (a zero vector scores 0)

// Sticky device-side error word at the start of every workspace.
struct WsHeader {
  unsigned int err;      // first quoka_status recorded by a kernel (0 = none)
  unsigned int where;    // kernel-specific detail (which wait expired)
  unsigned int pad[62];
};
static_assert(sizeof(WsHeader) == 256, "header keeps the workspace 256-byte aligned");

__device__ __forceinline__ void record_error(WsHeader* hdr, unsigned int code, unsigned int where) {
  if (hdr != nullptr && atomicCAS(&hdr->err, 0u, code) == 0u) hdr->where = where;
}

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation and, before touching global memory, waits
// until the kernels before it have completed (a no-op without the launch
// attribute).  A kernel releases its dependents either at its start (short or
// SM-filling kernels, so that the next kernel's launch and prologue overlap
// it) or as its last statement; never two in a row at the start, which would
// launch a whole chain of kernels whose CTAs then sit waiting on the SMs
// (released at the start everywhere, the step was 8% slower).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// pdl_wait(), then every pointer passed is laundered through an empty asm:
// loads from a `const __restrict__` pointer may be treated as invariant and
// scheduled above griddepcontrol.wait, where they would read what was there
// before the previous kernel wrote it; a load through the laundered value
// depends on the asm, which stays after the wait.
template <typename... P>
__device__ __forceinline__ void pdl_wait_for(P&... ptrs) {
  pdl_wait();
  (
      [&] {
        uintptr_t v = (uintptr_t)ptrs;
        asm volatile("" : "+l"(v)::"memory");
        ptrs = (P)v;
      }(),
      ...);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Monotone map of a float to uint32: a < b as floats  <=>  key(a) < key(b).
// -0.0 is folded onto +0.0 so that equal floats get equal keys.
__device__ __forceinline__ uint32_t order_key(float f) {
  if (f == 0.0f) f = 0.0f;
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The 12-bit histogram bin of a score, counted where the scores are produced
// so that the top-B select can start from the bin holding the B-th largest
// score.  Cosine scores lie in [-1, 1]: a fixed-point bin of width 1/2048
// (4096 bins over [-1, 1], the ends clamped), fine where the scores crowd
// together.  Other scores: the top 12 bits of order_key.  Both are
// non-decreasing in the score, with NaN in bin 0 for cosines.
__device__ __forceinline__ uint32_t score_bin(float s, bool cosine) {
  if (cosine) {
    const float t = __fmul_rn(__fadd_rn(s, 1.0f), 2048.0f);
    return t >= 0.0f ? (uint32_t)min(__float2int_rz(t), 4095) : 0u;
  }
  return order_key(s) >> 20;
}

// The float of an order key (inverse of order_key; -0.0 comes back as +0.0).
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// hist[bin] += 1 for every lane with `valid`; lanes of a warp with the same
// bin add once.  `hist` may be shared or global memory.  All 32 lanes call it.
__device__ __forceinline__ void hist_bin_add(unsigned int* hist, uint32_t bin, bool valid) {
  const uint32_t b = valid ? bin : 0xFFFFFFFFu;
  const unsigned peers = __match_any_sync(0xffffffffu, b);
  if (valid && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], (unsigned)__popc(peers));
}

// Exclusive prefix sum over a block of exactly blockDim.x threads (a multiple
// of 32, at most 1024).  `scratch` holds 32 ints.  Returns the exclusive
// prefix of `v`; *total receives the block sum.  Contains __syncthreads().
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarp ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    scratch[lane] = w;   // inclusive prefix over warps
  }
  __syncthreads();
  int warp_base = warp > 0 ? scratch[warp - 1] : 0;
  *total = scratch[nwarp - 1];
  int res = warp_base + x - v;
  __syncthreads();
  return res;
}

}  // namespace quoka
