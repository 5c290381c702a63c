// Tensor-core key scoring (bf16 keys, tcgen05 + TMA).
// Method: QUOKA paper summary, "Scoring via Cosine Similarity" and
// "Aggregation Across Queries and KV Groups"; QUOKA Explained, "Letting those
// queries score the history", "Why take the maximum".
//
// One pass over the history keys, each read from HBM once.  A CTA owns a
// contiguous range of 128-key tiles of one KV head.  Per tile:
//   D[128 keys x N_pad rows] = K_tile[128 x d] . (HI + LO)[N_pad x d]^T
// (tcgen05, fp32 in TMEM), the keys on the TMEM lanes, so the thread of a key
// reduces the maximum over the scoring rows from its own lane with no
// cross-thread step:   score[t] = max_r D[t, r] / |k_t|.
// HI + LO is the fp32 scoring row (a unit query for max pooling, the
// pre-aggregated row for mean pooling) split into two bf16 rows by
// k_build_operand; both MMA passes accumulate into the same TMEM columns, so
// the epilogue needs no per-row scale.  |k_t| comes from the key tile in
// shared memory, in fp32.
//
// Warp roles (192 threads): warp 0 issues TMA loads (operand once, then a ring
// of key tiles), warp 1 owns TMEM and issues the MMAs, warps 2-5 are the
// epilogue, one key per thread.  Shared memory is left to the tensor core's
// operand reads while an accumulator is being drained: the epilogue reads the
// key tile for |k|^2 before it waits for the accumulator, and between
// "accumulator full" and "accumulator free" it touches only TMEM and
// registers.  Every wait is bounded; on a timeout the CTA records
// QUOKA_ERR_TIMEOUT, lets in-flight copies and MMAs land, frees TMEM and exits.
#include "launch.h"
#include "tc_common.cuh"

namespace quoka {

namespace {

constexpr int kTileKeys = 128;
constexpr int kScoreThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kMaxStages = 8;

// Rows of one operand TMA box: it must divide NT = 2 * N_pad (<= 512) and be <= 256.
__host__ __device__ inline int op_box_rows(int NT) { return NT <= 256 ? NT : NT / 2; }

// Bounded wait done by lane 0 only, result broadcast, so the warp stays converged.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, WsHeader* hdr,
                                          unsigned where) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait(bar, parity, abort, hdr, where);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

struct ScoreSmem {
  uint64_t kv_full[kMaxStages];
  uint64_t kv_empty[kMaxStages];
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

// Maximum over n (32 or 64) TMEM columns of this thread's lane starting at
// taddr; columns at index >= lim (the operand's padding rows) are skipped.
template <int N>
__device__ __forceinline__ float tmem_max(uint32_t taddr, int lim, float m) {
  uint32_t v[N];
  if constexpr (N == 64) tc::tmem_ld64(taddr, v); else tc::tmem_ld32(taddr, v);
  if (lim < N) {
#pragma unroll
    for (int j = 0; j < N; ++j)
      if (j >= lim) v[j] = __float_as_uint(-INFINITY);
  }
  float m0 = m, m1 = -INFINITY;
#pragma unroll
  for (int j = 0; j < N / 4; ++j) {
    m0 = fmax3(m0, __uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]));
    m1 = fmax3(m1, __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
  }
  return fmaxf(m0, m1);
}

// Operand rows in shared memory: [HALVES][NT = 2 * N_pad][128 B]; row
// p * N_pad + r is pass p (0 = hi, 1 = lo) of scoring row r.
template <int D>
__global__ void __launch_bounds__(kScoreThreads, 1)
    k_score_tc(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap omap, int T_len, int R,
               int N_pad, int nst, int nacc, uint32_t tmem_cols, float* __restrict__ scores, WsHeader* hdr) {
  constexpr int HALVES = D / 64;
  constexpr uint32_t kHalfBytes = kTileKeys * 128;            // one 64-column half of a key tile
  constexpr uint32_t kStageBytes = HALVES * kHalfBytes;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int NT = 2 * N_pad;
  const uint32_t op_bytes = (uint32_t)HALVES * NT * 128;
  uint8_t* op_s = smem;                                         // [HALVES][NT][128 B]
  uint8_t* ktiles = smem + op_bytes;                            // [nst][HALVES][128][128 B]
  ScoreSmem* sm = reinterpret_cast<ScoreSmem*>(ktiles + (size_t)nst * kStageBytes);

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
      // The keys do not come from the previous kernel: start this CTA's first
      // tiles towards L2 while that kernel finishes.
      for (int it = 0; it < ntiles && it < nst; ++it)
        for (int hf = 0; hf < HALVES; ++hf) tc::tma_prefetch_l2_3d(&kmap, hf * 64, (tile0 + it) * kTileKeys, g);
      pdl_wait();                               // the operand comes from the previous kernel
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
        for (int nc = 0; nc < N_pad; nc += 256) {
          const int n_this = N_pad - nc < 256 ? N_pad - nc : 256;
          const uint32_t idesc = tc::idesc_bf16_f32(128, n_this, false);
#pragma unroll
          for (int p = 0; p < 2; ++p)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const int hf = kk >> 2, kin = kk & 3;
              const uint64_t adesc = tc::sw128_desc(a_base + hf * kHalfBytes + kin * 32, 16, 1024);
              const uint64_t bdesc =
                  tc::sw128_desc(b_base + ((uint32_t)hf * NT + p * N_pad + nc) * 128 + kin * 32, 16, 1024);
              tc::mma_ss(tmem + (uint32_t)(a * N_pad + nc), adesc, bdesc, idesc, (p | kk) > 0 ? 1u : 0u);
            }
        }
        tc::mma_commit(&sm->kv_empty[s]);
        tc::mma_commit(&sm->acc_full[a]);
      }
      tc::mma_commit(&sm->drain);        // completes once every MMA above has finished
      tc::mbar_drain(&sm->drain, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue: one key per thread
    const int quad = warp & 3;                      // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;               // key within the tile
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    bool alive = true;                              // false once a wait gave up (warp-uniform)
    for (int it = 0; it < ntiles; ++it) {
      const int s = it % nst, a = it % nacc;
      if (alive) alive = warp_wait(&sm->kv_full[s], (it / nst) & 1, abort, hdr, 0x105);
      float ss = 0.f;
      if (alive) {
        // |k|^2 from the tile (16-byte chunks; chunk c of row r sits at c ^ (r & 7))
        const uint8_t* rp = ktiles + (size_t)s * kStageBytes + (row >> 3) * 1024 + (row & 7) * 128;
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
        for (int chunk = 0; chunk < HALVES * 8; ++chunk) {
          const int hf = chunk >> 3, c = chunk & 7;
          const uint4 v = *reinterpret_cast<const uint4*>(rp + hf * kHalfBytes + ((c ^ (row & 7)) << 4));
          // bf16 pair -> two fp32 (exact: shift into the high half)
          float x = __uint_as_float(v.x << 16), y = __uint_as_float(v.x & 0xFFFF0000u);
          s0 = fmaf(x, x, s0);
          s1 = fmaf(y, y, s1);
          x = __uint_as_float(v.y << 16), y = __uint_as_float(v.y & 0xFFFF0000u);
          s2 = fmaf(x, x, s2);
          s3 = fmaf(y, y, s3);
          x = __uint_as_float(v.z << 16), y = __uint_as_float(v.z & 0xFFFF0000u);
          s0 = fmaf(x, x, s0);
          s1 = fmaf(y, y, s1);
          x = __uint_as_float(v.w << 16), y = __uint_as_float(v.w & 0xFFFF0000u);
          s2 = fmaf(x, x, s2);
          s3 = fmaf(y, y, s3);
        }
        ss = (s0 + s1) + (s2 + s3);
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm->kv_empty[s]);
      if (alive) alive = warp_wait(&sm->acc_full[a], (it / nacc) & 1, abort, hdr, 0x106);
      float m = -INFINITY;
      if (alive) {
        tc::tc_fence_after();
        const uint32_t base = tmem + lane_addr + (uint32_t)(a * N_pad);
        int c0 = 0;
        for (; c0 + 64 <= N_pad; c0 += 64) m = tmem_max<64>(base + c0, R - c0, m);
        if (c0 < N_pad) m = tmem_max<32>(base + c0, R - c0, m);
        tc::tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm->acc_empty[a]);
      const int t = (tile0 + it) * kTileKeys + row;
      if (alive && t < T_len) scores[(size_t)g * T_len + t] = m * (1.0f / fmaxf(sqrtf(ss), kNormEps));
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
// the epilogue reads TMEM 32 columns at a time.
int score_tc_pad_rows(int R) { return (R + 31) / 32 * 32; }

size_t score_tc_smem(int d, int N_pad, int nst) {
  return 1024 + (size_t)2 * (d / 64) * N_pad * 128 + (size_t)nst * (d / 64) * kTileKeys * 128 + sizeof(ScoreSmem);
}

cudaError_t launch_score_tc(int d, const void* K, int64_t head_stride, int H_kv, int T_len, const __nv_bfloat16* op_bf,
                            int R, float* scores, WsHeader* hdr, int num_sms, cudaStream_t st) {
  if (T_len == 0) return cudaSuccess;
  const int N_pad = score_tc_pad_rows(R);
  if (N_pad > 512) return cudaErrorInvalidValue;
  const size_t budget = 227 * 1024;
  int nst = kMaxStages;
  while (nst > 2 && score_tc_smem(d, N_pad, nst) > budget) --nst;
  const size_t smem = score_tc_smem(d, N_pad, nst);
  if (smem > budget) return cudaErrorInvalidValue;
  const int NT = 2 * N_pad;
  const int nacc = 2 * N_pad <= 512 ? 2 : 1;
  uint32_t cols = 32;
  while (cols < (uint32_t)(nacc * N_pad)) cols <<= 1;
  CUtensorMap kmap, omap;
  cudaError_t e = make_tmap_bf16_3d(&kmap, K, d, T_len, H_kv, (uint64_t)d * 2, (uint64_t)head_stride * 2, 64, 128);
  if (e != cudaSuccess) return e;
  e = make_tmap_bf16_3d(&omap, op_bf, d, (uint64_t)NT, H_kv, (uint64_t)d * 2, (uint64_t)NT * d * 2, 64,
                        op_box_rows(NT));
  if (e != cudaSuccess) return e;
  const int tiles_head = (T_len + kTileKeys - 1) / kTileKeys;
  int per_head = (num_sms + H_kv - 1) / H_kv;
  if (per_head > tiles_head) per_head = tiles_head;
  dim3 grid(per_head, H_kv);
  if (d == 64) {
    e = ensure_smem((const void*)k_score_tc<64>, smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(k_score_tc<64>, grid, dim3(kScoreThreads), smem, st, kmap, omap, T_len, R, N_pad, nst, nacc, cols,
                   scores, hdr);
    if (e != cudaSuccess) return e;
  } else {
    e = ensure_smem((const void*)k_score_tc<128>, smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(k_score_tc<128>, grid, dim3(kScoreThreads), smem, st, kmap, omap, T_len, R, N_pad, nst, nacc,
                   cols, scores, hdr);
    if (e != cudaSuccess) return e;
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace quoka
