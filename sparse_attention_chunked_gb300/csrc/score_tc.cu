// Tensor-core key scoring (bf16 keys, tcgen05 + TMA).
// Method: QUOKA paper summary, "Scoring via Cosine Similarity" and
// "Aggregation Across Queries and KV Groups"; QUOKA Explained, "Letting those
// queries score the history", "Why take the maximum".
//
// One pass over the history keys, each read from HBM once.  A CTA owns a
// contiguous range of 128-key tiles of one KV head.  Per tile:
//   D[128 keys x N rows] = K_tile[128 x d] . OP[N x d]^T   (tcgen05, fp32 in TMEM)
// with the keys on the TMEM lanes, so the epilogue thread of a key reduces the
// maximum over the scoring rows from its own lane with no cross-thread step:
//   score[t] = max_r (D[t, r] * scale[r]) / |k_t|.
// OP is the scoring operand built by k_build_operand: for max pooling the raw
// bf16 query rows (exact) with scale 1/|q|; for mean pooling the fp32
// pre-aggregated rows split as hi + lo bf16, both accumulated into the same
// TMEM columns (two MMA passes, scale 1).  |k_t| comes from the same shared
// memory tile, in fp32.
//
// Warp roles (576 threads): warp 0 issues TMA loads (operand once, then a ring
// of key tiles), warp 1 owns TMEM and issues the MMAs, warps 2-17 are the
// epilogue: four warps per TMEM lane quadrant, each reducing a quarter of the
// scoring rows and a quarter of the key's squared norm; the quarters meet in
// shared memory behind a named barrier of the 512 epilogue threads.  Every wait is bounded; on a timeout the
// CTA records QUOKA_ERR_TIMEOUT, lets in-flight copies and MMAs land, frees
// TMEM and exits.
#include "launch.h"
#include "tc_common.cuh"

namespace quoka {

namespace {

constexpr int kTileKeys = 128;
constexpr int kScoreThreads = 576;
constexpr int kEpiWarps = 16;
constexpr int kEpiParts = 4;

// Rows of one operand TMA box: it must divide N_pad (<= 512) and be <= 256.
__host__ __device__ inline int op_box_rows(int N_pad) { return N_pad <= 256 ? N_pad : N_pad / 2; }

// Bounded wait done by lane 0 only, result broadcast, so the warp stays converged.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, WsHeader* hdr,
                                          unsigned where) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait(bar, parity, abort, hdr, where);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

struct ScoreSmem {
  float red_max[2][kEpiParts][128];   // [tile parity][row quarter][key]
  float red_ss[2][kEpiParts][128];
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t op_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (a.x * b.x, a.y * b.y) and (a.x + b.x, a.y + b.y) as single packed instructions.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  unsigned long long pa, pb, pc;
  asm("mov.b64 %0, {%1, %2};" : "=l"(pa) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(pb) : "f"(b.x), "f"(b.y));
  asm("mul.f32x2 %0, %1, %2;" : "=l"(pc) : "l"(pa), "l"(pb));
  float2 c;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(c.x), "=f"(c.y) : "l"(pc));
  return c;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  unsigned long long pa, pb, pc;
  asm("mov.b64 %0, {%1, %2};" : "=l"(pa) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(pb) : "f"(b.x), "f"(b.y));
  asm("add.f32x2 %0, %1, %2;" : "=l"(pc) : "l"(pa), "l"(pb));
  float2 c;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(c.x), "=f"(c.y) : "l"(pc));
  return c;
}

// Operand rows in shared memory: [HALVES][NT][128 B], NT = passes * N_pad, so
// that one MMA with N = NT (in chunks of 256) covers every pass; pass p of row
// r is B row p * N_pad + r and lands in TMEM column p * N_pad + r.
template <int D>
__global__ void __maxnreg__(96)
    k_score_tc(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap omap,
               const float* __restrict__ op_scale, int T_len, int R, int N_pad, int passes, int nst, int nacc,
               uint32_t tmem_cols, float* __restrict__ scores, WsHeader* hdr) {
  constexpr int HALVES = D / 64;
  constexpr uint32_t kHalfBytes = kTileKeys * 128;            // one 64-column half of a key tile
  constexpr uint32_t kStageBytes = HALVES * kHalfBytes;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int NT = passes * N_pad;
  const uint32_t op_bytes = (uint32_t)HALVES * NT * 128;
  uint8_t* op_s = smem;                                         // [HALVES][NT][128 B]
  uint8_t* ktiles = smem + op_bytes;                            // [nst][HALVES][128][128 B]
  float* scale_s = reinterpret_cast<float*>(ktiles + (size_t)nst * kStageBytes);
  ScoreSmem* sm = reinterpret_cast<ScoreSmem*>(scale_s + N_pad);

  const int g = blockIdx.y;
  const int tiles_head = (T_len + kTileKeys - 1) / kTileKeys;
  const int per = (tiles_head + gridDim.x - 1) / gridDim.x;
  const int tile0 = blockIdx.x * per;
  const int ntiles = max(0, min(tiles_head, tile0 + per) - tile0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      tc::mbar_init(&sm->kv_full[s], 1);
      tc::mbar_init(&sm->kv_empty[s], 1 + kEpiWarps);
    }
    for (int a = 0; a < nacc; ++a) {
      tc::mbar_init(&sm->acc_full[a], 1);
      tc::mbar_init(&sm->acc_empty[a], kEpiWarps);
    }
    tc::mbar_init(&sm->op_full, 1);
    tc::mbar_init(&sm->drain, 1);
    sm->abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&sm->tmem_base, tmem_cols);
    tc::tmem_relinquish();
  }
  pdl_launch_dependents();
  pdl_wait();                                   // the operand and its scales come from the previous kernel
  for (int i = threadIdx.x; i < N_pad; i += blockDim.x) scale_s[i] = op_scale[(size_t)g * N_pad + i];
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile int* abort = &sm->abort;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && ntiles > 0) {
      tc::tma_prefetch_desc(&kmap);
      tc::tma_prefetch_desc(&omap);
      tc::mbar_arrive_expect_tx(&sm->op_full, op_bytes);
      const int nb = op_box_rows(NT);
      for (int hf = 0; hf < HALVES; ++hf)
        for (int rb = 0; rb < NT; rb += nb)
          tc::tma_load_3d(op_s + ((size_t)hf * NT + rb) * 128, &omap, &sm->op_full, hf * 64, rb, g);
      int issued = 0;
      for (int it = 0; it < ntiles; ++it) {
        const int s = it % nst;
        if (it >= nst && !tc::mbar_wait(&sm->kv_empty[s], ((it / nst) - 1) & 1, abort, hdr, 0x101)) break;
        tc::mbar_arrive_expect_tx(&sm->kv_full[s], kStageBytes);
        for (int hf = 0; hf < HALVES; ++hf)
          tc::tma_load_3d(ktiles + (size_t)s * kStageBytes + hf * kHalfBytes, &kmap, &sm->kv_full[s], hf * 64,
                          (tile0 + it) * kTileKeys, g);
        ++issued;
      }
      if (*abort) {   // let every copy already issued land before the CTA can exit
        tc::mbar_drain(&sm->op_full, 0);
        for (int it = issued - nst < 0 ? 0 : issued - nst; it < issued; ++it)
          tc::mbar_drain(&sm->kv_full[it % nst], (it / nst) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && ntiles > 0) {
      bool ok = tc::mbar_wait(&sm->op_full, 0, abort, hdr, 0x102);
      tc::tc_fence_after();
      const uint32_t b_base = tc::smem_u32(op_s);
      for (int it = 0; ok && it < ntiles; ++it) {
        const int s = it % nst, a = it % nacc;
        if (!tc::mbar_wait(&sm->kv_full[s], (it / nst) & 1, abort, hdr, 0x103)) break;
        if (it >= nacc && !tc::mbar_wait(&sm->acc_empty[a], ((it / nacc) - 1) & 1, abort, hdr, 0x104)) break;
        tc::tc_fence_after();
        const uint32_t a_base = tc::smem_u32(ktiles + (size_t)s * kStageBytes);
        for (int nc = 0; nc < NT; nc += 256) {
          const int n_this = NT - nc < 256 ? NT - nc : 256;
          const uint32_t idesc = tc::idesc_bf16_f32(128, n_this, false);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int hf = kk >> 2, kin = kk & 3;
            const uint64_t adesc = tc::sw128_desc(a_base + hf * kHalfBytes + kin * 32, 16, 1024);
            const uint64_t bdesc = tc::sw128_desc(b_base + ((uint32_t)hf * NT + nc) * 128 + kin * 32, 16, 1024);
            tc::mma_ss(tmem + (uint32_t)(a * NT + nc), adesc, bdesc, idesc, kk > 0 ? 1u : 0u);
          }
        }
        tc::mma_commit(&sm->kv_empty[s]);
        tc::mma_commit(&sm->acc_full[a]);
      }
      tc::mma_commit(&sm->drain);        // completes once every MMA above has finished
      tc::mbar_drain(&sm->drain, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue: one key per four threads
    const int quad = warp & 3;                      // TMEM lane quadrant this warp may access
    const int part = (warp - 2) >> 2;               // which quarter of the rows / of d
    const int row = quad * 32 + lane;               // key within the tile
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const int quarter = ((N_pad >> 2) + 31) & ~31;
    const int r_begin = min(N_pad, part * quarter), r_end = min(R, part == kEpiParts - 1 ? N_pad : (part + 1) * quarter);
    const bool mean_mode = passes == 2;
    bool alive = true;                              // false once a wait gave up (warp-uniform)
    for (int it = 0; it < ntiles; ++it) {
      const int s = it % nst, a = it % nacc, buf = it & 1;
      if (alive) alive = warp_wait(&sm->kv_full[s], (it / nst) & 1, abort, hdr, 0x105);
      float ss = 0.f;
      if (alive) {
        // |k|^2 over this part's quarter of d (16-byte chunks); chunk c of row r sits at c ^ (r & 7)
        const uint8_t* tile = ktiles + (size_t)s * kStageBytes;
        float ss0 = 0.f, ss1 = 0.f;
        constexpr int kChunks = HALVES * 8 / kEpiParts;   // 16-byte chunks of the row per part
#pragma unroll
        for (int cc = 0; cc < kChunks; ++cc) {
          const int chunk = part * kChunks + cc, hf = chunk >> 3, c = chunk & 7;
          const uint8_t* rp = tile + hf * kHalfBytes + (row >> 3) * 1024 + (row & 7) * 128;
          {
            const uint4 v = *reinterpret_cast<const uint4*>(rp + ((c ^ (row & 7)) << 4));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {           // bf16 pair -> two fp32 (exact: shift into the high half)
              const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
              ss0 = fmaf(lo, lo, ss0);
              ss1 = fmaf(hi, hi, ss1);
            }
          }
        }
        ss = ss0 + ss1;
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm->kv_empty[s]);
      if (alive) alive = warp_wait(&sm->acc_full[a], (it / nacc) & 1, abort, hdr, 0x106);
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (alive) {
        tc::tc_fence_after();
        for (int c0 = r_begin; c0 < r_end; c0 += 32) {
          uint32_t v[32];
          tc::tmem_ld32(tmem + lane_addr + (uint32_t)(a * NT + c0), v);
          if (mean_mode) {                           // hi + lo of the pre-aggregated row
            uint32_t w[32];
            tc::tmem_ld32(tmem + lane_addr + (uint32_t)(a * NT + N_pad + c0), w);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float2 s2 = add2(make_float2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])),
                                     make_float2(__uint_as_float(w[2 * j]), __uint_as_float(w[2 * j + 1])));
              v[2 * j] = __float_as_uint(s2.x);
              v[2 * j + 1] = __float_as_uint(s2.y);
            }
          } else {                                   // x 1/|q| of the raw query row
            const float4* sc = reinterpret_cast<const float4*>(scale_s + c0);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 q = sc[j];
              const float2 p0 = mul2(make_float2(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1])),
                                     make_float2(q.x, q.y));
              const float2 p1 = mul2(make_float2(__uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])),
                                     make_float2(q.z, q.w));
              v[4 * j] = __float_as_uint(p0.x);
              v[4 * j + 1] = __float_as_uint(p0.y);
              v[4 * j + 2] = __float_as_uint(p1.x);
              v[4 * j + 3] = __float_as_uint(p1.y);
            }
          }
          if (c0 + 32 > r_end) {                     // padding rows of the last chunk never win
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c0 + j >= r_end) v[j] = __float_as_uint(-INFINITY);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j)
            m4[j & 3] = fmax3(m4[j & 3], __uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
        }
        tc::tc_fence_before();
      }
      const float best = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm->acc_empty[a]);
      sm->red_max[buf][part][row] = best;
      sm->red_ss[buf][part][row] = ss;
      asm volatile("bar.sync 1, 512;" ::: "memory");   // the 16 epilogue warps
      if (part == 0 && alive) {
        const float mx = fmaxf(fmaxf(sm->red_max[buf][0][row], sm->red_max[buf][1][row]),
                               fmaxf(sm->red_max[buf][2][row], sm->red_max[buf][3][row]));
        const float rk = 1.0f / fmaxf(sqrtf((sm->red_ss[buf][0][row] + sm->red_ss[buf][1][row]) +
                                            (sm->red_ss[buf][2][row] + sm->red_ss[buf][3][row])), kNormEps);
        const int t = (tile0 + it) * kTileKeys + row;
        if (t < T_len) scores[(size_t)g * T_len + t] = mx * rk;
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, tmem_cols);
  }
}

}  // namespace

// Scoring rows padded to a multiple of 32: MMA N must be a multiple of 16 and
// the epilogue reads TMEM 32 columns at a time without crossing N_pad.
int score_tc_pad_rows(int R) { return (R + 31) / 32 * 32; }

size_t score_tc_smem(int d, int N_pad, int passes, int nst) {
  return 1024 + (size_t)passes * (d / 64) * N_pad * 128 + (size_t)nst * (d / 64) * kTileKeys * 128 +
         (size_t)N_pad * 4 + sizeof(ScoreSmem);
}

cudaError_t launch_score_tc(int d, const void* K, int64_t head_stride, int H_kv, int T_len, const __nv_bfloat16* op_bf,
                            const float* op_scale, int R, int passes, float* scores, WsHeader* hdr, int num_sms,
                            cudaStream_t st) {
  if (T_len == 0) return cudaSuccess;
  const int N_pad = score_tc_pad_rows(R);
  if (N_pad > 512) return cudaErrorInvalidValue;
  const size_t budget = 227 * 1024;
  int nst = 6;
  while (nst > 2 && score_tc_smem(d, N_pad, passes, nst) > budget) --nst;
  const size_t smem = score_tc_smem(d, N_pad, passes, nst);
  if (smem > budget) return cudaErrorInvalidValue;
  const int NT = passes * N_pad;
  if (NT > 512) return cudaErrorInvalidValue;
  const int nacc = 2 * NT <= 512 ? 2 : 1;
  uint32_t cols = 32;
  while (cols < (uint32_t)(nacc * NT)) cols <<= 1;
  CUtensorMap kmap, omap;
  cudaError_t e = make_tmap_bf16_3d(&kmap, K, d, T_len, H_kv, (uint64_t)d * 2, (uint64_t)head_stride * 2, 64, 128);
  if (e != cudaSuccess) return e;
  e = make_tmap_bf16_3d(&omap, op_bf, d, (uint64_t)passes * N_pad, H_kv, (uint64_t)d * 2,
                        (uint64_t)passes * N_pad * d * 2, 64, op_box_rows(NT));
  if (e != cudaSuccess) return e;
  const int tiles_head = (T_len + kTileKeys - 1) / kTileKeys;
  int per_head = (num_sms + H_kv - 1) / H_kv;
  if (per_head > tiles_head) per_head = tiles_head;
  dim3 grid(per_head, H_kv);
  if (d == 64) {
    e = ensure_smem((const void*)k_score_tc<64>, smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(k_score_tc<64>, grid, dim3(kScoreThreads), smem, st, kmap, omap, op_scale, T_len, R, N_pad, passes,
                   nst, nacc, cols, scores, hdr);
    if (e != cudaSuccess) return e;
  } else {
    e = ensure_smem((const void*)k_score_tc<128>, smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(k_score_tc<128>, grid, dim3(kScoreThreads), smem, st, kmap, omap, op_scale, T_len, R, N_pad, passes,
                   nst, nacc, cols, scores, hdr);
    if (e != cudaSuccess) return e;
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace quoka
