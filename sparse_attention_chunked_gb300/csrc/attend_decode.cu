// Attention for chunks of a few queries (decode: C = 1), split over the keys.
// Method: QUOKA paper summary, "Transformers and Attention" (softmax
// attention with a causal mask), "Chunked prefill" (the chunk attends to the
// earlier keys plus itself, causally), "QUOKA Method" (the reduced key set is
// fed to attention); QUOKA Explained, "From scores to a smaller KV set" (a
// kept key brings its value).
//
// With C small, a KV group has only G * C query rows, too few to fill a
// tensor-core tile or the GPU, while the keys number B_e + C.  So the keys are
// split into blocks of kDecKeys and every (block, KV group) is one CTA
// (flash-decoding): the CTA scores its keys against the group's rows, takes
// the block's softmax statistics (max m and sum l of exp2(s - m)) and the
// unnormalised output sum p . V, and writes them to the workspace; a second
// kernel merges the blocks of every row, rescaling each by exp2(m_b - M).
// The kept history rows are read straight from the cache through `sel` (no
// gathered copy), and every product and sum is an fp32 FMA on CUDA cores:
// with so few rows the step is bound by reading the kept K and V rows.
#include "common.cuh"
#include "launch.h"

namespace quoka {

namespace {

constexpr int kDecKeys = 64;       // keys per CTA
constexpr int kDecThreads = 256;

// Eight consecutive elements of a 16-byte load as fp32 (bf16: one load;
// fp32: the caller passes two).
__device__ __forceinline__ void widen(uint4 u, float (&x)[8]) {
  x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xFFFF0000u);
  x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xFFFF0000u);
  x[4] = __uint_as_float(u.z << 16); x[5] = __uint_as_float(u.z & 0xFFFF0000u);
  x[6] = __uint_as_float(u.w << 16); x[7] = __uint_as_float(u.w & 0xFFFF0000u);
}

// q . k over D elements: q fp32 in shared memory, k of type T in shared memory.
template <int D>
__device__ __forceinline__ float dot_row(const float* q, const __nv_bfloat16* k) {
  float s0 = 0.f, s1 = 0.f;
#pragma unroll 4
  for (int e = 0; e < D; e += 8) {
    float x[8];
    widen(*reinterpret_cast<const uint4*>(k + e), x);
    const float4 qa = *reinterpret_cast<const float4*>(q + e), qb = *reinterpret_cast<const float4*>(q + e + 4);
    s0 = fmaf(qa.x, x[0], s0); s1 = fmaf(qa.y, x[1], s1);
    s0 = fmaf(qa.z, x[2], s0); s1 = fmaf(qa.w, x[3], s1);
    s0 = fmaf(qb.x, x[4], s0); s1 = fmaf(qb.y, x[5], s1);
    s0 = fmaf(qb.z, x[6], s0); s1 = fmaf(qb.w, x[7], s1);
  }
  return s0 + s1;
}
template <int D>
__device__ __forceinline__ float dot_row(const float* q, const float* k) {
  float s0 = 0.f, s1 = 0.f;
#pragma unroll 4
  for (int e = 0; e < D; e += 4) {
    const float4 a = *reinterpret_cast<const float4*>(k + e), qa = *reinterpret_cast<const float4*>(q + e);
    s0 = fmaf(qa.x, a.x, s0); s1 = fmaf(qa.y, a.y, s1);
    s0 = fmaf(qa.z, a.z, s0); s1 = fmaf(qa.w, a.w, s1);
  }
  return s0 + s1;
}

// Rows of a group handled by one CTA: G * C when that is at most 32.
template <typename T, int D>
__global__ void __launch_bounds__(kDecThreads) k_attend_decode(
    const T* __restrict__ Q, const T* __restrict__ Kh, const T* __restrict__ Vh, int64_t h_stride,
    const int32_t* __restrict__ sel, int n_hist, int T_cache, const T* __restrict__ Kc, const T* __restrict__ Vc,
    int C, int G, float scale_log2, float* __restrict__ part_ml, float* __restrict__ part_o, WsHeader* hdr) {
  pdl_wait_for(Q, Kh, Vh, sel, Kc, Vc);
  constexpr int VEC = 16 / (int)sizeof(T);        // elements per 16-byte load
  constexpr int KP = D + VEC;                     // padded key row: conflict-free 16-byte reads across keys
  extern __shared__ __align__(16) float dsm[];
  float* Qs = dsm;                                // [32][D] fp32, scaled by scale * log2(e)
  float* Ps = Qs + 32 * D;                        // [32][kDecKeys + 1]
  T* Ks = reinterpret_cast<T*>(Ps + 32 * (kDecKeys + 1));   // [kDecKeys][KP], as stored in HBM
  T* Vs = Ks + kDecKeys * KP;                     // [kDecKeys][D]
  const int blk = blockIdx.x, g = blockIdx.y, n_blk = gridDim.x;
  const int R = G * C;
  const int j0 = blk * kDecKeys;
  const int n_keys = n_hist + C;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // The block's keys and values: kept history rows through sel, then the
  // chunk's rows.  The kept positions are fetched first, the query rows while
  // they are in flight, then every 16-byte K/V load of the block is issued
  // before the first is used: two dependent memory latencies in all.
  constexpr int NV = D / VEC;                                // loads per row
  constexpr int PER = kDecKeys * NV / kDecThreads;           // loads per thread, per tensor
  static_assert(kDecKeys * NV % kDecThreads == 0, "whole loads per thread");
  int64_t pos[PER];
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int j = j0 + (tid + u * kDecThreads) / NV;
    pos[u] = j < n_hist ? (sel != nullptr ? (int64_t)sel[(size_t)g * n_hist + j] : (int64_t)j) : -1;
  }
  // a kept position outside the cache is never read (its key and value stay zero rows)
  bool bad = false;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int j = j0 + (tid + u * kDecThreads) / NV;
    if (j < n_hist && (pos[u] < 0 || pos[u] >= T_cache)) {
      bad = true;
      pos[u] = -2;
    }
  }
  if (bad) record_error(hdr, 7u /* QUOKA_ERR_DEVICE */, (unsigned)(g * n_hist + j0));
  constexpr int QPER = 32 * D / kDecThreads;                 // query elements per thread (rows < R used)
  float qv[QPER];
#pragma unroll
  for (int u = 0; u < QPER; ++u) {
    const int i = tid + u * kDecThreads, r = i / D, e = i % D;
    qv[u] = r < R ? to_f32(Q[((size_t)(g * G + r / C) * C + r % C) * D + e]) : 0.f;
  }
  uint4 kr[PER], vr[PER];
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int i = tid + u * kDecThreads, jj = i / NV, e = (i % NV) * VEC;
    const int j = j0 + jj;
    kr[u] = vr[u] = make_uint4(0u, 0u, 0u, 0u);
    if (j < n_keys && pos[u] != -2) {
      const T *kp, *vp;
      if (j < n_hist) {
        kp = Kh + (size_t)g * h_stride + (size_t)pos[u] * D + e;
        vp = Vh + (size_t)g * h_stride + (size_t)pos[u] * D + e;
      } else {
        kp = Kc + ((size_t)g * C + (j - n_hist)) * D + e;
        vp = Vc + ((size_t)g * C + (j - n_hist)) * D + e;
      }
      kr[u] = *reinterpret_cast<const uint4*>(kp);
      vr[u] = *reinterpret_cast<const uint4*>(vp);
    }
  }
#pragma unroll
  for (int u = 0; u < QPER; ++u) Qs[tid + u * kDecThreads] = qv[u] * scale_log2;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int i = tid + u * kDecThreads, jj = i / NV, e = (i % NV) * VEC;
    *reinterpret_cast<uint4*>(Ks + jj * KP + e) = kr[u];
    *reinterpret_cast<uint4*>(Vs + jj * D + e) = vr[u];
  }
  __syncthreads();
  // scores: thread -> key jj = tid % 64 against rows r = tid / 64 + 4 i
  {
    const int jj = tid % kDecKeys, r0 = tid / kDecKeys;
    const int j = j0 + jj;
    for (int r = r0; r < R; r += kDecThreads / kDecKeys) {
      const float sc = dot_row<D>(Qs + r * D, Ks + jj * KP);
      // chunk key j - n_hist is visible to chunk row c iff it is not after it
      const bool ok = j < n_keys && (j < n_hist || j - n_hist <= r % C);
      Ps[r * (kDecKeys + 1) + jj] = ok ? sc : -INFINITY;
    }
  }
  __syncthreads();
  // per row: block max and sum of exp2(s - m); p stored back in place
  for (int r = warp; r < R; r += kDecThreads / 32) {
    float* pr = Ps + r * (kDecKeys + 1);
    const float a = pr[lane], b = pr[lane + 32];
    float m = fmaxf(a, b);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float pa = m == -INFINITY ? 0.f : exp2f(a - m);
    const float pb = m == -INFINITY ? 0.f : exp2f(b - m);
    float l = pa + pb;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    pr[lane] = pa;
    pr[lane + 32] = pb;
    if (lane == 0) {
      const size_t row = ((size_t)g * R + r) * n_blk + blk;
      part_ml[2 * row] = m;
      part_ml[2 * row + 1] = l;
    }
  }
  __syncthreads();
  // unnormalised output: thread -> column e = tid % D of rows r = tid / D + (256 / D) i
  {
    const int e = tid % D, rstep = kDecThreads / D;
    for (int r = tid / D; r < R; r += rstep) {
      const float* pr = Ps + r * (kDecKeys + 1);
      float o0 = 0.f, o1 = 0.f;
#pragma unroll 8
      for (int jj = 0; jj < kDecKeys; jj += 2) {
        o0 = fmaf(pr[jj], to_f32(Vs[jj * D + e]), o0);
        o1 = fmaf(pr[jj + 1], to_f32(Vs[(jj + 1) * D + e]), o1);
      }
      part_o[(((size_t)g * R + r) * n_blk + blk) * D + e] = o0 + o1;
    }
  }
  pdl_launch_dependents();   // dependents launch once this CTA is done
}

// One CTA per (group row): M = max_b m_b, w_b = 2^(m_b - M), L = sum_b l_b w_b,
// O = sum_b o_b w_b / L, lse = (M + log2 L) ln 2 in the units of the scaled
// logits.  The weights go to shared memory; then thread (e, s) sums column e
// over blocks s, s + S, ... (S = 256 / D), its loads independent of one
// another, and the S partial sums are added in shared memory.
constexpr int kMergeThreads = 256;

template <typename T, int D>
__global__ void __launch_bounds__(kMergeThreads) k_attend_decode_merge(const float* __restrict__ part_ml,
                                                                       const float* __restrict__ part_o, int n_blk,
                                                                       int C, int G, T* __restrict__ O,
                                                                       float* __restrict__ lse) {
  pdl_wait_for(part_ml, part_o);
  extern __shared__ float w_s[];                 // [n_blk]
  __shared__ float red[kMergeThreads / 32];
  __shared__ float part[kMergeThreads];
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* ml = part_ml + (size_t)row * n_blk * 2;
  float M = -INFINITY;
  for (int b = tid; b < n_blk; b += kMergeThreads) M = fmaxf(M, ml[2 * b]);
  M = warp_max(M);
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < kMergeThreads / 32; ++w) M = fmaxf(M, red[w]);
  __syncthreads();
  float L = 0.f;
  for (int b = tid; b < n_blk; b += kMergeThreads) {
    const float mb = ml[2 * b];
    const float w = mb == -INFINITY ? 0.f : exp2f(mb - M);
    w_s[b] = w;
    L = fmaf(ml[2 * b + 1], w, L);
  }
  L = warp_sum(L);
  if (lane == 0) red[warp] = L;
  __syncthreads();
  L = 0.f;
#pragma unroll
  for (int w = 0; w < kMergeThreads / 32; ++w) L += red[w];
  constexpr int S = kMergeThreads / D;
  const int e = tid % D, sub = tid / D;
  const float* ob = part_o + (size_t)row * n_blk * D + e;
  float a0 = 0.f, a1 = 0.f;
  int b = sub;
#pragma unroll 4
  for (; b + S < n_blk; b += 2 * S) {
    a0 = fmaf(ob[(size_t)b * D], w_s[b], a0);
    a1 = fmaf(ob[(size_t)(b + S) * D], w_s[b + S], a1);
  }
  if (b < n_blk) a0 = fmaf(ob[(size_t)b * D], w_s[b], a0);
  part[tid] = a0 + a1;
  __syncthreads();
  if (tid < D) {
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < S; ++k) acc += part[tid + k * D];
    // group row -> (head, chunk row)
    const int g = row / (G * C), r = row % (G * C);
    const int h = g * G + r / C, c = r % C;
    O[((size_t)h * C + c) * D + tid] = from_f32<T>(acc / L);
    if (lse != nullptr && tid == 0) lse[(size_t)h * C + c] = (M + log2f(L)) * 0.69314718055994531f;
  }
  pdl_launch_dependents();   // dependents launch once this CTA is done
}

size_t decode_smem(int d, int elt) {
  const int vec = 16 / elt;
  return ((size_t)32 * d + (size_t)32 * (kDecKeys + 1)) * 4 + ((size_t)kDecKeys * (d + vec) + (size_t)kDecKeys * d) * elt;
}

}  // namespace

bool attend_decode_fits(int C, int G) { return C * G <= 32; }

size_t attend_decode_ws_bytes(int d, int H_q, int C, int n_hist) {
  const size_t n_blk = (size_t)(n_hist + C + kDecKeys - 1) / kDecKeys;
  return (size_t)H_q * C * n_blk * (2 + (size_t)d) * 4;
}

cudaError_t launch_attend_decode(int dtype, int d, const void* Q, const void* Kh, const void* Vh, int64_t h_stride,
                                 const int32_t* sel, int n_hist, int T_cache, const void* Kc, const void* Vc, int H_q,
                                 int H_kv, int C, float scale, void* O, float* lse, float* part, WsHeader* hdr,
                                 cudaStream_t st) {
  const int G = H_q / H_kv;
  if (!attend_decode_fits(C, G)) return cudaErrorInvalidValue;
  const int n_blk = (n_hist + C + kDecKeys - 1) / kDecKeys;
  float* part_ml = part;
  float* part_o = part + (size_t)H_q * C * n_blk * 2;
  const float scale_log2 = scale * 1.4426950408889634f;
  const size_t smem = decode_smem(d, dtype == 0 ? 2 : 4);
  const dim3 grid(n_blk, H_kv), mgrid(H_q * C);
  const size_t msmem = (size_t)n_blk * 4;
  cudaError_t e;
#define QUOKA_DEC(T, DD)                                                                                          \
  do {                                                                                                            \
    e = ensure_smem((const void*)k_attend_decode<T, DD>, smem);                                                   \
    if (e == cudaSuccess)                                                                                         \
      e = launch_pdl(k_attend_decode<T, DD>, grid, dim3(kDecThreads), smem, st, (const T*)Q, (const T*)Kh,        \
                     (const T*)Vh, h_stride, sel, n_hist, T_cache, (const T*)Kc, (const T*)Vc, C, G, scale_log2,   \
                     part_ml, part_o, hdr);                                                                       \
    if (e == cudaSuccess) e = ensure_smem((const void*)k_attend_decode_merge<T, DD>, msmem);                     \
    if (e == cudaSuccess)                                                                                         \
      e = launch_pdl(k_attend_decode_merge<T, DD>, mgrid, dim3(kMergeThreads), msmem, st, (const float*)part_ml,  \
                     (const float*)part_o, n_blk, C, G, (T*)O, lse);                                              \
  } while (0)
  if (dtype == 0) {
    if (d == 64) QUOKA_DEC(__nv_bfloat16, 64); else QUOKA_DEC(__nv_bfloat16, 128);
  } else {
    if (d == 64) QUOKA_DEC(float, 64); else QUOKA_DEC(float, 128);
  }
#undef QUOKA_DEC
  if (e != cudaSuccess) return e;
  count_launches(2);
  return cudaGetLastError();
}

}  // namespace quoka
