// Tensor-core key scoring (bf16 keys, tcgen05 + TMA).
// Method: QUOKA paper summary, "Scoring via Cosine Similarity" and
// "Aggregation Across Queries and KV Groups"; QUOKA Explained, "Letting those
// queries score the history", "Why take the maximum".
//
// One pass over the history keys, each read from HBM once.  A CTA owns a
// contiguous range of 128-key tiles of one KV head.  Per tile:
//   D[128 keys x N rows] = K_tile[128 x d] . OP[N x d]^T
// (tcgen05, fp32 in TMEM), the keys on the TMEM lanes, so the threads of a key
// reduce the maximum over the scoring rows from their own lane:
//   score[t] = max_r (D[t, r] * s_r) / |k_t|.
// Operand forms, all exact to fp32 rounding:
//  * scaled (max pooling with more than 256 rows, where a hi/lo operand does
//    not fit shared memory): OP holds the selected query rows as they are
//    (bf16, exact) and s_r = 1 / |q_r| is applied per column in the
//    epilogue; one MMA pass.
//  * hi/lo: a row with no exact bf16 form (a unit query, a pre-aggregated
//    mean) is split by k_build_operand into hi + lo bf16 rows.  Up to 128
//    rows, one MMA of N = 2 N_pad covers [hi rows ; lo rows] and the
//    epilogue adds the two columns of a row; wider operands take two passes
//    into the same TMEM columns.  s_r = 1.
// The MMA reads its operands from shared memory at a fixed cost per
// instruction below N = 128, and shared-memory loads of the epilogue compete
// with those reads, which is why the forms above avoid a second pass and
// per-tile scale loads where they can.  |k_t| comes from the key tile in
// shared memory, in fp32 (or from the key-norm cache).
//
// Warp roles (320 threads): warp 0 issues TMA loads (operand once, then a ring
// of key tiles), warp 1 owns TMEM and issues the MMAs, warps 2-9 are the
// epilogue: the two warps of a TMEM lane quadrant share its 32 keys, each
// taking half of the columns (and half of |k|^2), and combine through shared
// memory.  The accumulator is a ring of two TMEM units of up to 256 columns;
// a tile with more than 256 scoring rows fills both in turn.  The epilogue
// copies a unit to registers and hands it back before its arithmetic, so the
// tensor core refills it meanwhile.  Every wait is bounded; on a timeout the
// CTA records QUOKA_ERR_TIMEOUT, lets in-flight copies and MMAs land, frees
// TMEM and exits.
#include "launch.h"
#include "tc_common.cuh"

namespace quoka {

namespace {

constexpr int kTileKeys = 128;
constexpr int kEpiWarps = 8;
constexpr int kScoreThreads = 64 + 32 * kEpiWarps;
constexpr int kMaxStages = 8;
constexpr int kUnitCols = 256;     // widest accumulator unit (one MMA's N)

// Operand forms (see the top of the file).
enum ScoreMode : int {
  kScaled = 0,      // raw rows, one pass, scales read from shared memory
  kHiLo = 1,        // hi/lo rows, two passes into the same columns
  kHiLoWide = 2,    // hi/lo rows, one MMA over 2 N_pad rows (N_pad <= 128)
};

// Rows of one operand TMA box: at most 256 and a divisor of NT (a multiple of 64).
__host__ __device__ inline int op_box_rows(int NT) { return NT % 256 == 0 ? 256 : NT % 128 == 0 ? 128 : 64; }

// Bounded wait done by lane 0 only, result broadcast, so the warp stays converged.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, WsHeader* hdr,
                                          unsigned where) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait(bar, parity, abort, hdr, where);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Barrier of the two epilogue warps of one TMEM lane quadrant (ids 1..4).
__device__ __forceinline__ void pair_sync(int quad) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + quad) : "memory");
}

struct ScoreSmem {
  uint64_t kv_full[kMaxStages];
  uint64_t kv_empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t op_full;
  uint64_t drain;
  unsigned int digit0[256];     // first radix digit of this CTA's scores (when asked for)
  float part_max[2][4][32];     // upper warp of a quadrant -> lower warp, by tile parity
  float part_ss[2][4][32];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (a0, a1) += (b0, b1) elementwise, one packed fp32 add.
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  uint64_t x, y, z;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b0), "f"(b1));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(z) : "l"(x), "l"(y));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(z));
}

// (a0, a1) * (b0, b1) elementwise, one packed fp32 multiply.
__device__ __forceinline__ void fmul2(float& a0, float& a1, float b0, float b1) {
  uint64_t x, y, z;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b0), "f"(b1));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(z) : "l"(x), "l"(y));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(z));
}

// Maximum over HW (32, 64, 96 or 128) TMEM columns of this thread's lane
// starting at taddr, each multiplied by its row scale sc[j] when SCALED;
// columns at index >= lim (the operand's padding rows) are skipped.  The
// columns are copied to registers and the accumulator unit is handed back
// (arrive on `empty`) before any arithmetic, so the scale loads from shared
// memory and the maximum run while the tensor core refills the unit.
template <int HW, bool SCALED, bool MASK>
__device__ __forceinline__ float max_cols(const uint32_t (&v)[HW], const float* sc, int lim, float m) {
  float m0 = m, m1 = -INFINITY;
#pragma unroll
  for (int j4 = 0; j4 < HW / 4; ++j4) {
    float x0 = __uint_as_float(v[4 * j4]), x1 = __uint_as_float(v[4 * j4 + 1]);
    float x2 = __uint_as_float(v[4 * j4 + 2]), x3 = __uint_as_float(v[4 * j4 + 3]);
    if constexpr (SCALED) {
      const float4 s4 = reinterpret_cast<const float4*>(sc)[j4];   // same address in every lane
      fmul2(x0, x1, s4.x, s4.y);
      fmul2(x2, x3, s4.z, s4.w);
    }
    if constexpr (MASK) {
      if (4 * j4 >= lim) x0 = -INFINITY;
      if (4 * j4 + 1 >= lim) x1 = -INFINITY;
      if (4 * j4 + 2 >= lim) x2 = -INFINITY;
      if (4 * j4 + 3 >= lim) x3 = -INFINITY;
    }
    m0 = fmax3(m0, x0, x1);
    m1 = fmax3(m1, x2, x3);
  }
  return fmaxf(m0, m1);
}

template <int HW, bool SCALED>
__device__ __forceinline__ float drain_max(uint32_t taddr, const float* sc, int lim, float m, uint64_t* empty,
                                           int lane) {
  uint32_t v[HW];
  if constexpr (HW == 128) {
    tc::tmem_ld128(taddr, v);
  } else if constexpr (HW == 96) {
    tc::tmem_ld64(taddr, v);
    tc::tmem_ld32(taddr + 64, v + 64);
  } else if constexpr (HW == 64) {
    tc::tmem_ld64(taddr, v);
  } else {
    tc::tmem_ld32(taddr, v);
  }
  tc::tc_fence_before();
  __syncwarp();
  if (lane == 0) tc::mbar_arrive(empty);
  return lim < HW ? max_cols<HW, SCALED, true>(v, sc, lim, m) : max_cols<HW, SCALED, false>(v, sc, lim, m);
}

// Copies HW consecutive TMEM columns of this thread's lane to registers.
template <int HW>
__device__ __forceinline__ void tmem_cols(uint32_t taddr, uint32_t (&v)[HW]) {
  static_assert(HW == 32 || HW == 64, "32 or 64 columns");
  if constexpr (HW == 64) tc::tmem_ld64(taddr, v);
  else tc::tmem_ld32(taddr, v);
}

// hi/lo in one MMA: this thread's HW rows have their hi dot products at
// hi_addr and their lo dot products at lo_addr; score row j = hi_j + lo_j.
template <int HW, bool MASK>
__device__ __forceinline__ float max_hilo(const uint32_t (&a)[HW], const uint32_t (&b)[HW], int lim, float m) {
  float m0 = m, m1 = -INFINITY;
#pragma unroll
  for (int j4 = 0; j4 < HW / 4; ++j4) {
    float x0 = __uint_as_float(a[4 * j4]), x1 = __uint_as_float(a[4 * j4 + 1]);
    float x2 = __uint_as_float(a[4 * j4 + 2]), x3 = __uint_as_float(a[4 * j4 + 3]);
    add2(x0, x1, __uint_as_float(b[4 * j4]), __uint_as_float(b[4 * j4 + 1]));
    add2(x2, x3, __uint_as_float(b[4 * j4 + 2]), __uint_as_float(b[4 * j4 + 3]));
    if constexpr (MASK) {
      if (4 * j4 >= lim) x0 = -INFINITY;
      if (4 * j4 + 1 >= lim) x1 = -INFINITY;
      if (4 * j4 + 2 >= lim) x2 = -INFINITY;
      if (4 * j4 + 3 >= lim) x3 = -INFINITY;
    }
    m0 = fmax3(m0, x0, x1);
    m1 = fmax3(m1, x2, x3);
  }
  return fmaxf(m0, m1);
}

template <int HW>
__device__ __forceinline__ float drain_hilo(uint32_t hi_addr, uint32_t lo_addr, int lim, float m, uint64_t* empty,
                                            int lane) {
  uint32_t a[HW], b[HW];
  tmem_cols<HW>(hi_addr, a);
  tmem_cols<HW>(lo_addr, b);
  tc::tc_fence_before();
  __syncwarp();
  if (lane == 0) tc::mbar_arrive(empty);
  return lim < HW ? max_hilo<HW, true>(a, b, lim, m) : max_hilo<HW, false>(a, b, lim, m);
}


// Operand rows in shared memory: [HALVES][NT][128 B] with NT = N_pad (scaled)
// or 2 N_pad (hi/lo: row p * N_pad + r is part p of scoring row r).  Column
// chunk c of a tile covers scoring rows [c * cw, c * cw + width) and goes to
// accumulator unit q & 1, q counting (tile, chunk) pairs; in the kHiLoWide
// form the single chunk is [hi columns ; lo columns], cw = 2 N_pad.
template <int D, int MODE>
__global__ void __launch_bounds__(kScoreThreads, 1)
    k_score_tc(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap omap,
               const float* __restrict__ op_scale, int T_len, int R, int N_pad, int nst, int cw,
               uint32_t tmem_cols, KeyScale ks, float* __restrict__ scores, unsigned* __restrict__ hist0,
               WsHeader* hdr) {
  constexpr int HALVES = D / 64;
  constexpr bool SCALED = MODE == kScaled;
  constexpr int NPASS = SCALED ? 1 : 2;          // operand rows per scoring row
  constexpr int NMMA = MODE == kHiLo ? 2 : 1;     // MMA passes into the same columns
  constexpr uint32_t kHalfBytes = kTileKeys * 128;            // one 64-column half of a key tile
  constexpr uint32_t kStageBytes = HALVES * kHalfBytes;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int NT = NPASS * N_pad;
  const int nch = MODE == kHiLoWide ? 1 : (N_pad + cw - 1) / cw;
  const uint32_t op_bytes = (uint32_t)HALVES * NT * 128;
  uint8_t* op_s = smem;                                         // [HALVES][NT][128 B]
  uint8_t* ktiles = smem + op_bytes;                            // [nst][HALVES][128][128 B]
  float* sc_s = reinterpret_cast<float*>(ktiles + (size_t)nst * kStageBytes);   // [N_pad] row scales
  ScoreSmem* sm = reinterpret_cast<ScoreSmem*>(sc_s + (SCALED ? N_pad : 0));

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
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&sm->acc_full[a], 1);
      tc::mbar_init(&sm->acc_empty[a], kEpiWarps);
    }
    tc::mbar_init(&sm->op_full, 1);
    tc::mbar_init(&sm->drain, 1);
    sm->abort = 0;
    tc::fence_mbar_init();
  }
  for (int b = threadIdx.x; b < 256; b += blockDim.x) sm->digit0[b] = 0;
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
      tc::mbar_arrive_expect_tx(&sm->op_full, op_bytes + (SCALED ? (uint32_t)N_pad * 4 : 0u));
      const int nb = op_box_rows(NT);
      for (int hf = 0; hf < HALVES; ++hf)
        for (int rb = 0; rb < NT; rb += nb)
          tc::tma_load_3d(op_s + ((size_t)hf * NT + rb) * 128, &omap, &sm->op_full,
                          hf * 64, rb, g);
      if constexpr (SCALED) tc::bulk_load(sc_s, op_scale + (size_t)g * N_pad, (uint32_t)N_pad * 4, &sm->op_full);
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
      // descriptors: a base descriptor plus (byte offset >> 4) in its address field
      // (shared addresses are below 256 KB, so the 14-bit field never carries)
      const uint64_t b_desc = tc::sw128_desc(tc::smem_u32(op_s), 16, 1024);
      for (int it = 0; ok && it < ntiles; ++it) {
        const int s = it % nst;
        if (!(ok = tc::mbar_wait(&sm->kv_full[s], (it / nst) & 1, abort, hdr, 0x103))) break;
        const uint64_t a_desc = tc::sw128_desc(tc::smem_u32(ktiles + (size_t)s * kStageBytes), 16, 1024);
        for (int c = 0; c < nch; ++c) {
          const int q = it * nch + c, u = q & 1;
          if (q >= 2 && !(ok = tc::mbar_wait(&sm->acc_empty[u], ((q >> 1) - 1) & 1, abort, hdr, 0x104))) break;
          tc::tc_fence_after();
          const int c0 = c * cw, width = MODE == kHiLoWide ? NT : min(cw, N_pad - c0);
          const uint32_t idesc = tc::idesc_bf16_f32(128, width, false);
#pragma unroll
          for (int p = 0; p < NMMA; ++p)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const int hf = kk >> 2, kin = kk & 3;
              const uint64_t adesc = a_desc + (uint64_t)((hf * kHalfBytes + kin * 32) >> 4);
              const uint64_t bdesc = b_desc + (uint64_t)((((uint32_t)hf * NT + p * N_pad + c0) * 128 + kin * 32) >> 4);
              tc::mma_ss(tmem + (uint32_t)(u * cw), adesc, bdesc, idesc, (p | kk) > 0 ? 1u : 0u);
            }
          if (c == nch - 1) tc::mma_commit(&sm->kv_empty[s]);
          tc::mma_commit(&sm->acc_full[u]);
        }
      }
      tc::mma_commit(&sm->drain);        // completes once every MMA above has finished
      tc::mbar_drain(&sm->drain, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;                      // TMEM lane quadrant this warp may access
    const int half = (warp - 2) >> 2;               // which half of the columns (and of |k|^2)
    const int row = quad * 32 + lane;               // key within the tile
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    bool alive = ntiles > 0;                        // false once a wait gave up (warp-uniform)
    if constexpr (SCALED) {
      if (alive) alive = warp_wait(&sm->op_full, 0, abort, hdr, 0x107);   // sc_s is in place
    }
    int q = 0;
    for (int it = 0; it < ntiles; ++it) {
      const int s = it % nst;
      if (alive) alive = warp_wait(&sm->kv_full[s], (it / nst) & 1, abort, hdr, 0x105);
      float ss = 0.f, rk = 1.f;
      const int t = (tile0 + it) * kTileKeys + row;
      if (ks.key_norm && ks.k_inv != nullptr && half == 0)   // the key-norm cache: one load, issued early
        rk = t < T_len ? ks.k_inv[(size_t)g * ks.k_inv_stride + t] : 0.f;
      if (alive && ks.key_norm && ks.k_inv == nullptr) {
        // this half's share of |k|^2 (16-byte chunks; chunk c of row r sits at c ^ (r & 7))
        const uint8_t* rp = ktiles + (size_t)s * kStageBytes + (row >> 3) * 1024 + (row & 7) * 128;
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
        for (int j = 0; j < HALVES * 4; ++j) {
          const int chunk = half * HALVES * 4 + j;
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
      float m = -INFINITY;
      for (int c = 0; c < nch; ++c, ++q) {
        const int u = q & 1;
        if (alive) alive = warp_wait(&sm->acc_full[u], (q >> 1) & 1, abort, hdr, 0x106);
        if (alive) {
          tc::tc_fence_after();
          uint64_t* empty = &sm->acc_empty[u];
          const uint32_t unit = tmem + lane_addr + (uint32_t)(u * cw);
          if constexpr (MODE == kHiLoWide) {
            // scoring rows [half * hw, half * hw + hw): hi at those columns, lo N_pad further
            const int hw = N_pad >> 1, col = half * hw;
            const uint32_t hi = unit + (uint32_t)col, lo = hi + (uint32_t)N_pad;
            if (hw == 64) m = drain_hilo<64>(hi, lo, R - col, m, empty, lane);
            else m = drain_hilo<32>(hi, lo, R - col, m, empty, lane);
          } else {
            const int c0 = c * cw, hw = min(cw, N_pad - c0) >> 1;   // this warp's columns: 32, 64, 96 or 128
            const int col = c0 + half * hw;
            const uint32_t base = unit + (uint32_t)(half * hw);
            const float* sc = sc_s + col;
            if (hw == 128) m = drain_max<128, SCALED>(base, sc, R - col, m, empty, lane);
            else if (hw == 96) m = drain_max<96, SCALED>(base, sc, R - col, m, empty, lane);
            else if (hw == 64) m = drain_max<64, SCALED>(base, sc, R - col, m, empty, lane);
            else m = drain_max<32, SCALED>(base, sc, R - col, m, empty, lane);
          }
        } else {
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&sm->acc_empty[u]);
        }
      }
      // the quadrant's upper warp hands its half to the lower warp, which writes the score
      const int buf = it & 1;
      if (half == 1) {
        sm->part_max[buf][quad][lane] = m;
        sm->part_ss[buf][quad][lane] = ss;
      }
      pair_sync(quad);
      if (half == 0) {
        m = fmaxf(m, sm->part_max[buf][quad][lane]);
        ss += sm->part_ss[buf][quad][lane];
        if (ks.key_norm && ks.k_inv == nullptr) rk = 1.0f / fmaxf(sqrtf(ss), kNormEps);
        if (alive && t < T_len) scores[(size_t)g * T_len + t] = m * rk;
        if (hist0 != nullptr) digit0_add(sm->digit0, order_key(m * rk), alive && t < T_len);
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, tmem_cols);
  }
  if (hist0 != nullptr)   // this CTA's share of the head's first-digit histogram
    for (int b = threadIdx.x; b < 256; b += blockDim.x)
      if (sm->digit0[b] != 0) atomicAdd(&hist0[(size_t)g * 256 + b], sm->digit0[b]);
}

template <int D, int MODE>
cudaError_t launch_one(dim3 grid, size_t smem, cudaStream_t st, const CUtensorMap& kmap, const CUtensorMap& omap,
                       const float* op_scale, int T_len, int R, int N_pad, int nst, int cw, uint32_t cols,
                       KeyScale ks, float* scores, unsigned* hist0, WsHeader* hdr) {
  cudaError_t e = ensure_smem((const void*)k_score_tc<D, MODE>, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_score_tc<D, MODE>, grid, dim3(kScoreThreads), smem, st, kmap, omap, op_scale, T_len, R, N_pad,
                    nst, cw, cols, ks, scores, hist0, hdr);
}

}  // namespace

// Scoring rows padded to a multiple of 64: each epilogue warp then reads its
// half of a column chunk from TMEM 32 columns at a time.
int score_tc_pad_rows(int R) { return (R + 63) / 64 * 64; }

size_t score_tc_smem(int d, int N_pad, int npass, int nst) {
  return 1024 + (size_t)npass * (d / 64) * N_pad * 128 + (size_t)nst * (d / 64) * kTileKeys * 128 +
         (npass == 1 ? (size_t)N_pad * 4 : 0) + sizeof(ScoreSmem);
}

cudaError_t launch_score_tc(int d, const void* K, int64_t head_stride, int H_kv, int T_len, const __nv_bfloat16* op_bf,
                            const float* op_scale, int R, KeyScale ks, float* scores, unsigned* hist0,
                            WsHeader* hdr, int num_sms, cudaStream_t st) {
  if (T_len == 0) return cudaSuccess;
  const int N_pad = score_tc_pad_rows(R);
  const int npass = op_scale != nullptr ? 1 : 2;
  if (N_pad > 512) return cudaErrorInvalidValue;
  const size_t budget = 227 * 1024;
  int nst = kMaxStages;
  while (nst > 2 && score_tc_smem(d, N_pad, npass, nst) > budget) --nst;
  const size_t smem = score_tc_smem(d, N_pad, npass, nst);
  if (smem > budget) return cudaErrorInvalidValue;
  const int NT = npass * N_pad;
  // operand form: see ScoreMode
  const int mode = npass == 1 ? kScaled : (N_pad <= 128 ? kHiLoWide : kHiLo);
  const int cw = mode == kHiLoWide ? 2 * N_pad : (N_pad < kUnitCols ? N_pad : kUnitCols);   // accumulator unit width
  uint32_t cols = 32;
  while (cols < (uint32_t)(2 * cw)) cols <<= 1;
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
#define QUOKA_SCORE_LAUNCH(DD, MM)                                                                             \
  launch_one<DD, MM>(grid, smem, st, kmap, omap, op_scale, T_len, R, N_pad, nst, cw, cols, ks, scores, hist0, hdr)
  if (d == 64)
    e = mode == kScaled ? QUOKA_SCORE_LAUNCH(64, kScaled)
        : mode == kHiLo ? QUOKA_SCORE_LAUNCH(64, kHiLo)
                        : QUOKA_SCORE_LAUNCH(64, kHiLoWide);
  else
    e = mode == kScaled ? QUOKA_SCORE_LAUNCH(128, kScaled)
        : mode == kHiLo ? QUOKA_SCORE_LAUNCH(128, kHiLo)
                        : QUOKA_SCORE_LAUNCH(128, kHiLoWide);
#undef QUOKA_SCORE_LAUNCH
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace quoka
