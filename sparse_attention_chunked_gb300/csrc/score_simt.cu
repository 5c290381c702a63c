// Scoring operand and the CUDA-core scoring kernel.
// Method: QUOKA paper summary, "Scoring via Cosine Similarity" and
// "Aggregation Across Queries and KV Groups"; QUOKA Explained, "Letting those
// queries score the history", "Why take the maximum", "A wrinkle:
// grouped-query attention".
#include "common.cuh"
#include "launch.h"

namespace quoka {

// One warp per scoring row; grid.x covers N_pad >= R rows (padding rows of
// the tensor-core copy repeat row 0, so they never change a maximum).  Row r of
// KV group g:
//   MAX : r = k * n + i  -> query head h = g*G + k, position q_idx[h, i];
//         fp32 row q / |q|.
//   MEAN: r = i          -> position q_idx[g, i];
//         fp32 row (1/G) sum_k q_k / |q_k| over the group's heads (not
//         re-normalised).
// Tensor-core copy of either: hi = bf16(row) in pass 0 and lo = bf16(row - hi)
// in pass 1 (hi + lo carries the fp32 row to about 2^-16 relative).
// Layouts: op_f32 [H_kv, R, D]; op_bf [H_kv, 2, N_pad, D].
// One block per scoring row.  Row r of group g is the weighted sum over its
// (head, token) pairs of the (unit) query rows:
//   mode 1:           pairs (head k, token i), r = k * n + i, weight 1;
//   mode 1 + qmean:   r = k, pairs (head k, every selected token), weight 1/n;
//   mode 0:           r = i, pairs (every head of g, token i), weight 1/G;
//   mode 0 + qmean:   r = 0, every (head, token) of g, weight 1/(G n).
// A row of one pair is one warp's work; rows that average many pairs get a
// block of kOpWarps warps, warp w taking pairs w, w + kOpWarps, ..., and the
// warps' sums are added in shared memory.
constexpr int kOpWarps = 8;

template <typename T, int D>
__global__ void __launch_bounds__(32 * kOpWarps) k_build_operand(const T* __restrict__ Q,
                                                                 const int32_t* __restrict__ q_idx, int C, int G,
                                                                 int n, OperandSpec spec, int R,
                                                                 float* __restrict__ op_f32,
                                                                 __nv_bfloat16* __restrict__ op_bf,
                                                                 float* __restrict__ op_scale,
                                                                 unsigned* __restrict__ hist) {
  pdl_launch_dependents();   // early: the scorer's prologue overlaps this short kernel
  pdl_wait_for(Q, q_idx);
  if (hist != nullptr && blockIdx.x == 0)   // the scorer that follows accumulates into it
    for (int b = threadIdx.x; b < kScoreHistBins; b += blockDim.x) hist[(size_t)blockIdx.y * kScoreHistBins + b] = 0;
  constexpr int E = D / 32;
  const int g = blockIdx.y, r_out = blockIdx.x, N_pad = gridDim.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int npass = op_scale != nullptr ? 1 : 2;
  if (r_out >= R && op_bf == nullptr) return;   // padding rows exist in the tensor-core copy only
  const int r = r_out < R ? r_out : 0;          // a padding row repeats row 0
  // the (head, token) pairs of row r: heads [k0, k1) of the group, tokens [i0, i1) of the selection
  int k0, k1, i0, i1;
  if (spec.mode == 1) {
    k0 = spec.qmean ? r : r / n;
    i0 = spec.qmean ? 0 : r % n;
    i1 = spec.qmean ? n : i0 + 1;
  } else {
    k0 = 0;
    i0 = spec.qmean ? 0 : r;
    i1 = spec.qmean ? n : r + 1;
  }
  k1 = spec.mode == 1 ? k0 + 1 : G;
  const int ni = i1 - i0, pairs = (k1 - k0) * ni;
  float acc[E];
#pragma unroll
  for (int j = 0; j < E; ++j) acc[j] = 0.f;
  float x[E], inv = 1.f;
  for (int p = warp; p < pairs; p += nwarps) {
    const int h = g * G + k0 + p / ni, i = i0 + p % ni;
    const int c = q_idx != nullptr ? q_idx[(size_t)(spec.mode == 1 ? h : g) * n + i] : i;   // NULL: every position
    const T* q = Q + ((size_t)h * C + c) * D;
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < E; ++j) {
      x[j] = to_f32(q[lane + 32 * j]);
      ss = fmaf(x[j], x[j], ss);
    }
    inv = spec.unit ? 1.0f / fmaxf(sqrtf(warp_sum(ss)), kNormEps) : 1.f;
#pragma unroll
    for (int j = 0; j < E; ++j) acc[j] = fmaf(x[j], inv, acc[j]);
  }
  if (nwarps > 1) {
    __shared__ float part[kOpWarps][D];
#pragma unroll
    for (int j = 0; j < E; ++j) part[warp][lane + 32 * j] = acc[j];
    __syncthreads();
    if (warp != 0) return;
#pragma unroll
    for (int j = 0; j < E; ++j) {
      float t = 0.f;
      for (int w = 0; w < nwarps; ++w) t += part[w][lane + 32 * j];
      acc[j] = t;
    }
  }
  if (pairs > 1) {
    const float w = 1.0f / (float)pairs;
#pragma unroll
    for (int j = 0; j < E; ++j) acc[j] *= w;
  }
  if (op_bf != nullptr && npass == 1) {   // one (head, token) pair: the query row itself and its scale
#pragma unroll
    for (int j = 0; j < E; ++j) op_bf[((size_t)g * N_pad + r_out) * D + lane + 32 * j] = __float2bfloat16_rn(x[j]);
    if (lane == 0) op_scale[(size_t)g * N_pad + r_out] = inv;
  }
  if (op_bf != nullptr && npass == 2) {
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(acc[j]);
      const __nv_bfloat16 lo = __float2bfloat16_rn(acc[j] - __bfloat162float(hi));
      op_bf[(((size_t)g * 2 + 0) * N_pad + r_out) * D + lane + 32 * j] = hi;
      op_bf[(((size_t)g * 2 + 1) * N_pad + r_out) * D + lane + 32 * j] = lo;
    }
  }
  if (op_f32 != nullptr && r_out < R) {
#pragma unroll
    for (int j = 0; j < E; ++j) op_f32[((size_t)g * R + r) * D + lane + 32 * j] = acc[j];
  }
}

// One thread per history key: its row is held in registers, the scoring rows
// stream through shared memory 32 at a time; score = max_r(r . k) / |k|.
template <typename T, int D>
__global__ void __launch_bounds__(128) k_score_simt(const T* __restrict__ K, int64_t head_stride, int T_len,
                                                    const float* __restrict__ op_f32, int R, KeyScale ks,
                                                    float* __restrict__ scores, unsigned* __restrict__ hist) {
  pdl_wait_for(K, op_f32);
  const int g = blockIdx.y;
  const int t = blockIdx.x * 128 + threadIdx.x;
  __shared__ float rows[32][D];
  float k[D];
  float ss = 0.f;
  if (t < T_len) {
    // the key row with 16-byte loads, all issued before the first is used
    const uint4* kp = reinterpret_cast<const uint4*>(K + (size_t)g * head_stride + (size_t)t * D);
    constexpr int NV = D * (int)sizeof(T) / 16;
    uint4 raw[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) raw[v] = kp[v];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const uint32_t w[4] = {raw[v].x, raw[v].y, raw[v].z, raw[v].w};
      if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          k[8 * v + 2 * j] = __uint_as_float(w[j] << 16);
          k[8 * v + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) k[4 * v + j] = __uint_as_float(w[j]);
      }
    }
#pragma unroll
    for (int e = 0; e < D; ++e) ss = fmaf(k[e], k[e], ss);
  } else {
#pragma unroll
    for (int e = 0; e < D; ++e) k[e] = 0.f;
  }
  const float rk = !ks.key_norm ? 1.0f
                  : ks.k_inv != nullptr ? (t < T_len ? ks.k_inv[(size_t)g * ks.k_inv_stride + t] : 0.f)
                                        : 1.0f / fmaxf(sqrtf(ss), kNormEps);
  float best = -INFINITY;
  const float* opg = op_f32 + (size_t)g * R * D;
  for (int r0 = 0; r0 < R; r0 += 32) {
    const int nr = min(32, R - r0);
    __syncthreads();
    for (int i = threadIdx.x; i < nr * D; i += 128) rows[i / D][i % D] = opg[(size_t)r0 * D + i];
    __syncthreads();
    for (int rr = 0; rr < nr; ++rr) {
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < D; ++e) dot = fmaf(k[e], rows[rr][e], dot);
      best = fmaxf(best, dot);
    }
  }
  if (t < T_len) scores[(size_t)g * T_len + t] = best * rk;
  if (hist != nullptr)   // the score's 12-bit bin, straight into the head's histogram
    hist_bin_add(hist + (size_t)g * kScoreHistBins, score_bin(best * rk, ks.key_norm), t < T_len);
  pdl_launch_dependents();   // dependents launch once this CTA is done
}

// Few scoring rows (R <= 8, e.g. a decode step's G unit queries): LPK lanes
// share one key row, each holding D / LPK of its elements, so a warp load
// reads LPK * 16 contiguous bytes of each of 32 / LPK rows; the scoring rows'
// matching elements stay in the lane's registers for the whole block.  Per
// key a lane does (R + 1) * D / LPK FMAs (R dot products and |k|^2), then
// log2(LPK) xor-shuffle steps per value give every lane of the group the
// totals; the group's first lane writes the score.  U key slots per warp are
// loaded before any is used.
template <typename T, int D, int LPK, int RMAX>
__global__ void __launch_bounds__(256) k_score_rows(const T* __restrict__ K, int64_t head_stride, int T_len,
                                                    const float* __restrict__ op_f32, int R, KeyScale ks,
                                                    float* __restrict__ scores, unsigned* __restrict__ hist) {
  constexpr int EPC = 16 / (int)sizeof(T);            // elements per 16-byte chunk
  constexpr int NCH = D / EPC;                        // chunks per key row
  constexpr int VPL = NCH / LPK;                      // chunks per lane per key
  constexpr int KPW = 32 / LPK;                       // keys per warp per slot
  constexpr int U = 4;                                // slots per warp
  constexpr int KPB = 8 * KPW * U;                    // keys per block
  static_assert(NCH % LPK == 0, "LPK must divide the chunks of a row");
  pdl_wait_for(K, op_f32);   // the scoring rows come from the previous kernel
  const int g = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane % LPK, kw = lane / LPK;
  // this lane's elements of every scoring row: chunk sub + LPK * v
  float q[RMAX][VPL][EPC];
  const float* opg = op_f32 + (size_t)g * R * D;
#pragma unroll
  for (int r = 0; r < RMAX; ++r)
#pragma unroll
    for (int v = 0; v < VPL; ++v)
#pragma unroll
      for (int j = 0; j < EPC; ++j) q[r][v][j] = r < R ? opg[(size_t)r * D + (sub + LPK * v) * EPC + j] : 0.f;
  // the key rows of the warp's U slots, every load issued before any is used
  const int t0 = blockIdx.x * KPB + warp * KPW * U;
  uint4 raw[U][VPL];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int t = t0 + u * KPW + kw;
    const uint4* kp = reinterpret_cast<const uint4*>(K + (size_t)g * head_stride + (size_t)t * D);
#pragma unroll
    for (int v = 0; v < VPL; ++v) raw[u][v] = t < T_len ? kp[sub + LPK * v] : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int t = t0 + u * KPW + kw;
    float dot[RMAX], ss = 0.f;
#pragma unroll
    for (int r = 0; r < RMAX; ++r) dot[r] = 0.f;
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      const uint32_t w[4] = {raw[u][v].x, raw[u][v].y, raw[u][v].z, raw[u][v].w};
      float x[EPC];
      if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {   // bf16 pair -> two fp32 (exact: shift into the high half)
          x[2 * j] = __uint_as_float(w[j] << 16);
          x[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = __uint_as_float(w[j]);
      }
#pragma unroll
      for (int j = 0; j < EPC; ++j) {
        ss = fmaf(x[j], x[j], ss);
#pragma unroll
        for (int r = 0; r < RMAX; ++r) dot[r] = fmaf(x[j], q[r][v][j], dot[r]);
      }
    }
#pragma unroll
    for (int o = LPK / 2; o > 0; o >>= 1) {
      ss += __shfl_xor_sync(0xffffffffu, ss, o);
#pragma unroll
      for (int r = 0; r < RMAX; ++r) dot[r] += __shfl_xor_sync(0xffffffffu, dot[r], o);
    }
    float best = dot[0];
#pragma unroll
    for (int r = 1; r < RMAX; ++r)
      if (r < R) best = fmaxf(best, dot[r]);
    const bool valid = t < T_len;
    const float rk = !ks.key_norm ? 1.0f
                    : ks.k_inv != nullptr ? (valid ? ks.k_inv[(size_t)g * ks.k_inv_stride + t] : 0.f)
                                          : 1.0f / fmaxf(sqrtf(ss), kNormEps);
    const float sc = best * rk;
    if (sub == 0 && valid) scores[(size_t)g * T_len + t] = sc;
    if (hist != nullptr) hist_bin_add(hist + (size_t)g * kScoreHistBins, score_bin(sc, ks.key_norm), sub == 0 && valid);
  }
  pdl_launch_dependents();   // dependents launch once this CTA is done
}

cudaError_t launch_build_operand(int dtype, int d, const void* Q, const int32_t* q_idx, int H_kv, int C, int G,
                                 int n, OperandSpec spec, int N_pad, float* op_f32, __nv_bfloat16* op_bf,
                                 float* op_scale, unsigned* hist, cudaStream_t st) {
  const int R = spec.mode == 1 ? (spec.qmean ? G : G * n) : (spec.qmean ? 1 : n);
  if (op_scale != nullptr && (spec.mode != 1 || spec.qmean || dtype != 0 || op_bf == nullptr))
    return cudaErrorInvalidValue;
  dim3 grid(op_bf != nullptr ? N_pad : R, H_kv);
  // rows that average several (head, token) pairs get a block of warps, single-pair rows one warp
  const int pairs = (spec.mode == 1 ? 1 : G) * (spec.qmean ? n : 1);
  const dim3 block(pairs > 1 ? 32 * kOpWarps : 32);
  cudaError_t e;
  if (dtype == 0) {
    if (d == 64)
      e = launch_pdl(k_build_operand<__nv_bfloat16, 64>, grid, block, 0, st, (const __nv_bfloat16*)Q, q_idx, C, G, n,
                     spec, R, op_f32, op_bf, op_scale, hist);
    else
      e = launch_pdl(k_build_operand<__nv_bfloat16, 128>, grid, block, 0, st, (const __nv_bfloat16*)Q, q_idx, C, G,
                     n, spec, R, op_f32, op_bf, op_scale, hist);
  } else {
    if (d == 64)
      e = launch_pdl(k_build_operand<float, 64>, grid, block, 0, st, (const float*)Q, q_idx, C, G, n, spec, R,
                     op_f32, op_bf, op_scale, hist);
    else
      e = launch_pdl(k_build_operand<float, 128>, grid, block, 0, st, (const float*)Q, q_idx, C, G, n, spec, R,
                     op_f32, op_bf, op_scale, hist);
  }
  count_launches(1);
  return e;
}

template <typename T, int D, int LPK, int RMAX>
static cudaError_t launch_rows(const void* K, int64_t head_stride, int H_kv, int T_len, const float* op_f32, int R,
                               KeyScale ks, float* scores, unsigned* hist, cudaStream_t st) {
  constexpr int KPB = 8 * (32 / LPK) * 4;
  return launch_pdl(k_score_rows<T, D, LPK, RMAX>, dim3((T_len + KPB - 1) / KPB, H_kv), dim3(256), 0, st,
                    (const T*)K, head_stride, T_len, op_f32, R, ks, scores, hist);
}

// Lanes per key row of k_score_rows: 8 up to 4 rows; 16 up to 8 rows where a
// row has 16 or more 16-byte chunks (the lane then keeps 64 operand values).
template <typename T, int D>
static cudaError_t launch_rows_r(const void* K, int64_t head_stride, int H_kv, int T_len, const float* op_f32, int R,
                                 KeyScale ks, float* scores, unsigned* hist, cudaStream_t st) {
  constexpr int NCH = D * (int)sizeof(T) / 16;
  if (R <= 4) return launch_rows<T, D, 8, 4>(K, head_stride, H_kv, T_len, op_f32, R, ks, scores, hist, st);
  return launch_rows<T, D, (NCH >= 16 ? 16 : 8), 8>(K, head_stride, H_kv, T_len, op_f32, R, ks, scores, hist, st);
}

cudaError_t launch_score_simt(int dtype, int d, const void* K, int64_t head_stride, int H_kv, int T_len,
                              const float* op_f32, int R, KeyScale ks, float* scores, unsigned* hist,
                              cudaStream_t st) {
  if (T_len == 0) return cudaSuccess;
  if (R <= kScoreRowsMax) {
    cudaError_t e;
    if (dtype == 0)
      e = d == 64 ? launch_rows_r<__nv_bfloat16, 64>(K, head_stride, H_kv, T_len, op_f32, R, ks, scores, hist, st)
                  : launch_rows_r<__nv_bfloat16, 128>(K, head_stride, H_kv, T_len, op_f32, R, ks, scores, hist, st);
    else
      e = d == 64 ? launch_rows_r<float, 64>(K, head_stride, H_kv, T_len, op_f32, R, ks, scores, hist, st)
                  : launch_rows_r<float, 128>(K, head_stride, H_kv, T_len, op_f32, R, ks, scores, hist, st);
    count_launches(1);
    return e;
  }
  dim3 grid((T_len + 127) / 128, H_kv);
  cudaError_t e;
  if (dtype == 0) {
    if (d == 64)
      e = launch_pdl(k_score_simt<__nv_bfloat16, 64>, grid, dim3(128), 0, st, (const __nv_bfloat16*)K, head_stride, T_len, op_f32, R, ks, scores, hist);
    else
      e = launch_pdl(k_score_simt<__nv_bfloat16, 128>, grid, dim3(128), 0, st, (const __nv_bfloat16*)K, head_stride, T_len, op_f32, R, ks, scores, hist);
  } else {
    if (d == 64)
      e = launch_pdl(k_score_simt<float, 64>, grid, dim3(128), 0, st, (const float*)K, head_stride, T_len, op_f32, R, ks, scores, hist);
    else
      e = launch_pdl(k_score_simt<float, 128>, grid, dim3(128), 0, st, (const float*)K, head_stride, T_len, op_f32, R, ks, scores, hist);
  }
  count_launches(1);
  return e;
}

}  // namespace quoka
