// Tensor-core key scoring (bf16 keys, tcgen05 + TMA).
// Method: QUOKA paper summary, "Scoring via Cosine Similarity" and
// "Aggregation Across Queries and KV Groups"; QUOKA Explained, "Letting those
// queries score the history", "Why take the maximum".
//
// One pass over the history keys, each read from HBM once.  A CTA owns a
// contiguous range of 128-key tiles of one KV head.  Per tile:
//   D[128 keys x N rows] = K_tile[128 x d] . OP[N x d]^T
// (tcgen05, fp32 in TMEM), the keys on the TMEM lanes, and
//   score[t] = max_r (D[t, r] * s_r) / |k_t|.
// Operand forms, all exact to fp32 rounding:
//  * scaled (max pooling): OP holds the selected query rows as they are
//    (bf16, exact) and s_r = 1 / |q_r|; one MMA pass.
//  * hi/lo: a row with no exact bf16 form (a pre-aggregated mean, a mean over
//    tokens) is split by k_build_operand into hi + lo bf16 rows; up to 128
//    rows one MMA of N = 2 N_pad covers [hi rows ; lo rows] and the epilogue
//    adds the two columns of a row, wider operands take two MMA passes into
//    the same columns.  s_r = 1.
// Padding rows (up to a multiple of 64) repeat row 0, so they never change a
// maximum and the epilogue needs no mask.
//
// Warp roles (320 threads): warp 0 issues TMA loads (operand once, then a ring
// of key stages), warp 1 owns TMEM and issues the MMAs, warps 2-9 are two
// epilogue groups of four warps (one per TMEM lane quadrant).  A tile's
// accumulator of up to 256 columns is one TMEM unit; the two groups take
// alternate tiles, each with its own unit, so one group's epilogue overlaps
// the other's and the tensor core refills a unit while the other is read.  A
// tile wider than 256 columns (more than 256 scaled rows) is two units, one per
// group, and the two partial maxima meet in shared memory.
//
// The epilogue reads TMEM with the 16x256b shape: a thread holds 4 keys of
// its quadrant (lanes t/4 + 8i) and 2 of every 8 columns (2 (t%4) + {0, 1}),
// so each thread needs the scales of a quarter of the columns only and keeps
// them in registers for the whole kernel; the 4 threads of a key combine
// their maxima with two shuffles.  |k_t|^2 is read from the key stage in
// shared memory (the 4 threads of a key take a quarter of its 16-byte chunks
// each) or comes from the key-norm cache.
//
// With `hist` the epilogue also counts every score's 12-bit bin (score_bin:
// fixed-point for cosines), where the top-B select starts, in a shared
// histogram, added to the head's global histogram at the end.  Every wait is
// bounded; on a timeout the CTA records QUOKA_ERR_TIMEOUT, lets in-flight
// copies and MMAs land, frees TMEM and exits.
#include "launch.h"
#include "tc_common.cuh"

namespace quoka {

namespace {

constexpr int kTileKeys = 128;
constexpr int kEpiWarps = 8;
constexpr int kScoreThreads = 64 + 32 * kEpiWarps;
constexpr int kMaxStages = 6;
constexpr int kUnitCols = 256;     // widest accumulator unit (one MMA's N)
constexpr int kPiece = 32;         // columns per epilogue TMEM read
constexpr int kMaxPieces = kUnitCols / kPiece;

// Operand forms (see the top of the file).
enum ScoreMode : int {
  kScaled = 0,      // raw rows, one pass, per-row scales
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
  float part_max[2][4][32];     // group 1 -> group 0 of a quadrant, by tile parity (two-unit tiles)
  float part_ss[2][4][32];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (a0, a1) *= (b0, b1) elementwise, one packed fp32 multiply.
__device__ __forceinline__ void fmul2(float& a0, float& a1, float b0, float b1) {
  uint64_t x, y, z;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b0), "f"(b1));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(z) : "l"(x), "l"(y));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(z));
}

// (a0, a1) += (b0, b1) elementwise, one packed fp32 add.
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  uint64_t x, y, z;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b0), "f"(b1));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(z) : "l"(x), "l"(y));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(z));
}

// 32 columns of the 32 lanes of this warp's quadrant: two 16x256b.x4 reads
// (lanes +0..15 into v[0..15], lanes +16..31 into v[16..31]).
__device__ __forceinline__ void load_piece(uint32_t taddr, uint32_t (&v)[32]) {
  tc::tmem_ld16x256b_x4(taddr, v);
  tc::tmem_ld16x256b_x4(taddr + (16u << 16), v + 16);
}

// Running maxima of this thread's 4 keys over one piece.  Key i of the thread
// is lane t/4 + 8i of the quadrant: v[16 (i >> 1) + 4j + 2 (i & 1) + e] holds
// its column 8j + 2 (t % 4) + e of the piece.
template <bool SCALED>
__device__ __forceinline__ void piece_max(const uint32_t (&v)[32], const float* sc, float (&m)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int b = 16 * (i >> 1) + 2 * (i & 1);
    float x[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = __uint_as_float(v[b + 4 * j]);
      x[2 * j + 1] = __uint_as_float(v[b + 4 * j + 1]);
      if constexpr (SCALED) fmul2(x[2 * j], x[2 * j + 1], sc[2 * j], sc[2 * j + 1]);
    }
    m[i] = fmax3(m[i], fmax3(x[0], x[1], x[2]), fmax3(x[3], x[4], fmax3(x[5], x[6], x[7])));
  }
}

// hi/lo in one MMA: the same layout for the hi columns (a) and lo columns (b).
__device__ __forceinline__ void piece_max_hilo(const uint32_t (&a)[32], const uint32_t (&b)[32], float (&m)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int o = 16 * (i >> 1) + 2 * (i & 1);
    float x[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = __uint_as_float(a[o + 4 * j]);
      x[2 * j + 1] = __uint_as_float(a[o + 4 * j + 1]);
      add2(x[2 * j], x[2 * j + 1], __uint_as_float(b[o + 4 * j]), __uint_as_float(b[o + 4 * j + 1]));
    }
    m[i] = fmax3(m[i], fmax3(x[0], x[1], x[2]), fmax3(x[3], x[4], fmax3(x[5], x[6], x[7])));
  }
}

// Operand rows in shared memory: [HALVES][NT][128 B] with NT = N_pad (scaled)
// or 2 N_pad (hi/lo: row p * N_pad + r is part p of scoring row r).  Chunk c
// of a tile (nch chunks of cw columns) covers scoring rows [c cw, c cw + cw)
// and chunk q (counting (tile, chunk) pairs) goes to accumulator unit q & 1
// and to epilogue group q & 1; in the kHiLoWide form the one chunk is
// [hi columns ; lo columns], cw = 2 N_pad.
template <int D, int MODE>
__global__ void __launch_bounds__(kScoreThreads, 1)
    k_score_tc(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap omap,
               const float* __restrict__ op_scale, int T_len, int N_pad, int nst, int nch, int cw,
               uint32_t tmem_cols, KeyScale ks, float* __restrict__ scores, unsigned* __restrict__ hist,
               WsHeader* hdr) {
  pdl_launch_dependents();   // early: the top-B CTAs take SMs as this kernel's CTAs finish
  constexpr int HALVES = D / 64;
  constexpr bool SCALED = MODE == kScaled;
  constexpr int NPASS = SCALED ? 1 : 2;          // operand rows per scoring row
  constexpr int NMMA = MODE == kHiLo ? 2 : 1;     // MMA passes into the same columns
  constexpr uint32_t kHalfBytes = kTileKeys * 128;            // one 64-column half of a key tile
  constexpr uint32_t kStageBytes = HALVES * kHalfBytes;
  constexpr int kChunks = D / 32;                             // 16-byte chunks of a key row per thread
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int NT = NPASS * N_pad;
  const uint32_t op_bytes = (uint32_t)HALVES * NT * 128;
  uint8_t* op_s = smem;                                         // [HALVES][NT][128 B]
  uint8_t* ktiles = smem + op_bytes;                            // [nst][HALVES][128][128 B]
  float* sc_s = reinterpret_cast<float*>(ktiles + (size_t)nst * kStageBytes);   // [N_pad] row scales
  unsigned* hist_s = reinterpret_cast<unsigned*>(sc_s + (SCALED ? N_pad : 0));  // [4096] when hist
  ScoreSmem* sm = reinterpret_cast<ScoreSmem*>(hist_s + (hist != nullptr ? kScoreHistBins : 0));

  const int g = blockIdx.y;
  const int tiles_head = (T_len + kTileKeys - 1) / kTileKeys;
  // tiles [tile0, tile0 + ntiles): the head's tiles split as evenly as possible
  const int tile0 = (int)((long long)blockIdx.x * tiles_head / gridDim.x);
  const int ntiles = (int)((long long)(blockIdx.x + 1) * tiles_head / gridDim.x) - tile0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      tc::mbar_init(&sm->kv_full[s], 1);
      // the MMAs, plus the epilogue warps when they read |k|^2 from the stage
      tc::mbar_init(&sm->kv_empty[s], 1 + (ks.key_norm && ks.k_inv == nullptr ? (nch == 1 ? 4 : 8) : 0));
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&sm->acc_full[a], 1);
      tc::mbar_init(&sm->acc_empty[a], 4);
    }
    tc::mbar_init(&sm->op_full, 1);
    tc::mbar_init(&sm->drain, 1);
    sm->abort = 0;
    tc::fence_mbar_init();
  }
  if (hist != nullptr)
    for (int b = threadIdx.x; b < kScoreHistBins; b += blockDim.x) hist_s[b] = 0;
  if (warp == 1) {
    tc::tmem_alloc(&sm->tmem_base, tmem_cols);
    tc::tmem_relinquish();
  }
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
          tc::tma_load_3d(op_s + ((size_t)hf * NT + rb) * 128, &omap, &sm->op_full, hf * 64, rb, g);
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
      const int width = MODE == kHiLoWide ? NT : cw;
      const uint32_t idesc = tc::idesc_bf16_f32(128, width, false);
      for (int it = 0; ok && it < ntiles; ++it) {
        const int s = it % nst;
        if (!(ok = tc::mbar_wait(&sm->kv_full[s], (it / nst) & 1, abort, hdr, 0x103))) break;
        const uint64_t a_desc = tc::sw128_desc(tc::smem_u32(ktiles + (size_t)s * kStageBytes), 16, 1024);
        for (int c = 0; c < nch; ++c) {
          const int q = it * nch + c, u = q & 1;
          if (q >= 2 && !(ok = tc::mbar_wait(&sm->acc_empty[u], ((q >> 1) - 1) & 1, abort, hdr, 0x104))) break;
          tc::tc_fence_after();
          const int c0 = c * cw;
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
    const int grp = (warp - 2) >> 2;                // epilogue group = accumulator unit
    const int quad = warp & 3;                      // TMEM lane quadrant this warp may access
    const int kr = lane >> 2, c4 = lane & 3;        // keys kr + 8i of the quadrant; column slice c4
    const uint32_t unit = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(grp * cw);
    const int chunk = nch == 2 ? grp : 0;           // the columns this group reads: [chunk cw, chunk cw + cw)
    const int npieces = (MODE == kHiLoWide ? N_pad : cw) / kPiece;
    // |k|^2 chunks: a key row's 16-byte chunks j of this thread (of kChunks per thread); with two
    // units per tile the groups split them
    const int j_lo = nch == 2 ? grp * (kChunks / 2) : 0;
    const int j_hi = nch == 2 ? j_lo + kChunks / 2 : kChunks;
    const bool norm_from_keys = ks.key_norm && ks.k_inv == nullptr;
    bool alive = ntiles > 0;                        // false once a wait gave up (warp-uniform)
    float sc[SCALED ? kMaxPieces * 8 : 1];          // this thread's row scales (8 columns per piece)
    if constexpr (SCALED) {
      if (alive) alive = warp_wait(&sm->op_full, 0, abort, hdr, 0x107);   // sc_s is in place
#pragma unroll
      for (int p = 0; p < kMaxPieces; ++p)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int col = chunk * cw + p * kPiece + 8 * j + 2 * c4;
          const bool in = p < npieces && alive;
          sc[8 * p + 2 * j] = in ? sc_s[col] : 0.f;
          sc[8 * p + 2 * j + 1] = in ? sc_s[col + 1] : 0.f;
        }
    }
    const int step = nch == 1 ? 2 : 1;
    for (int it = nch == 1 ? grp : 0; it < ntiles; it += step) {
      const int s = it % nst;
      // this thread's output key: i = c4, i.e. lane kr + 8 c4 of the quadrant
      const int t = (tile0 + it) * kTileKeys + quad * 32 + kr + 8 * c4;
      float rk = 1.f;
      if (ks.key_norm && ks.k_inv != nullptr)      // the key-norm cache: one load, issued early
        rk = t < T_len ? ks.k_inv[(size_t)g * ks.k_inv_stride + t] : 0.f;
      if (alive && norm_from_keys) alive = warp_wait(&sm->kv_full[s], (it / nst) & 1, abort, hdr, 0x105);
      float ss[4] = {0.f, 0.f, 0.f, 0.f};
      if (alive && norm_from_keys) {
        const uint8_t* stage = ktiles + (size_t)s * kStageBytes;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = quad * 32 + kr + 8 * i;
          const uint8_t* rp = stage + (row >> 3) * 1024 + (row & 7) * 128;
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int j = 0; j < kChunks; ++j) {
            if (j < j_lo || j >= j_hi) continue;
            const int gc = 8 * (j >> 1) + ((4 * (j & 1) + c4) ^ (4 * (kr & 1)));
            const int hf = gc >> 3, c = gc & 7;
            const uint4 v = *reinterpret_cast<const uint4*>(rp + hf * kHalfBytes + ((c ^ (row & 7)) << 4));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
              s0 = fmaf(lo, lo, s0);
              s1 = fmaf(hi, hi, s1);
            }
          }
          ss[i] = s0 + s1;
        }
      }
      if (norm_from_keys) {   // done with the key stage
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm->kv_empty[s]);
      }
      const int q = it * nch + chunk;
      float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (alive) alive = warp_wait(&sm->acc_full[grp], (q >> 1) & 1, abort, hdr, 0x106);
      if (alive) {
        tc::tc_fence_after();
#pragma unroll
        for (int p = 0; p < kMaxPieces; ++p) {
          if (p >= npieces) break;
          const bool last = p == npieces - 1;
          if constexpr (MODE == kHiLoWide) {
            uint32_t a[32], b[32];
            load_piece(unit + (uint32_t)(p * kPiece), a);
            load_piece(unit + (uint32_t)(N_pad + p * kPiece), b);
            tc::tmem_wait_ld_32(a);
            tc::tmem_wait_ld_32(b);
            if (last) {
              tc::tc_fence_before();
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(&sm->acc_empty[grp]);
            }
            piece_max_hilo(a, b, m);
          } else {
            uint32_t v[32];
            load_piece(unit + (uint32_t)(p * kPiece), v);
            tc::tmem_wait_ld_32(v);
            if (last) {   // the unit is copied out: the tensor core may refill it
              tc::tc_fence_before();
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(&sm->acc_empty[grp]);
            }
            piece_max<SCALED>(v, SCALED ? sc + 8 * p : nullptr, m);
          }
        }
      } else {
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm->acc_empty[grp]);
      }
      // the 4 threads of a key (lanes 4 kr .. 4 kr + 3) combine their column slices
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        m[i] = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], 1));
        m[i] = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], 2));
        ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], 1);
        ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], 2);
      }
      float my_m = c4 == 0 ? m[0] : c4 == 1 ? m[1] : c4 == 2 ? m[2] : m[3];
      float my_ss = c4 == 0 ? ss[0] : c4 == 1 ? ss[1] : c4 == 2 ? ss[2] : ss[3];
      if (nch == 2) {   // group 1 hands its half of the columns (and of |k|^2) to group 0
        const int buf = it & 1;
        if (grp == 1) {
          sm->part_max[buf][quad][kr + 8 * c4] = my_m;
          sm->part_ss[buf][quad][kr + 8 * c4] = my_ss;
        }
        pair_sync(quad);
        if (grp == 0) {
          my_m = fmaxf(my_m, sm->part_max[buf][quad][kr + 8 * c4]);
          my_ss += sm->part_ss[buf][quad][kr + 8 * c4];
        }
      }
      if (nch == 1 || grp == 0) {
        if (norm_from_keys) rk = 1.0f / fmaxf(sqrtf(my_ss), kNormEps);
        else if (!ks.key_norm) rk = 1.f;
        const float val = my_m * rk;
        if (alive && t < T_len) scores[(size_t)g * T_len + t] = val;
        if (hist != nullptr) hist_bin_add(hist_s, score_bin(val, ks.key_norm), alive && t < T_len);
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, tmem_cols);
  }
  if (hist != nullptr)   // this CTA's share of the head's histogram
    for (int b = threadIdx.x; b < kScoreHistBins; b += blockDim.x)
      if (hist_s[b] != 0) atomicAdd(&hist[(size_t)g * kScoreHistBins + b], hist_s[b]);
}

template <int D, int MODE>
cudaError_t launch_one(dim3 grid, size_t smem, cudaStream_t st, const CUtensorMap& kmap, const CUtensorMap& omap,
                       const float* op_scale, int T_len, int N_pad, int nst, int nch, int cw, uint32_t cols,
                       KeyScale ks, float* scores, unsigned* hist, WsHeader* hdr) {
  cudaError_t e = ensure_smem((const void*)k_score_tc<D, MODE>, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_score_tc<D, MODE>, grid, dim3(kScoreThreads), smem, st, kmap, omap, op_scale, T_len, N_pad, nst,
                    nch, cw, cols, ks, scores, hist, hdr);
}

}  // namespace

// Scoring rows padded to a multiple of 64 (whole 32-column epilogue pieces,
// also when a tile's columns are split into two units).
int score_tc_pad_rows(int R) { return (R + 63) / 64 * 64; }

size_t score_tc_smem(int d, int N_pad, int npass, int nst, bool hist) {
  return 1024 + (size_t)npass * (d / 64) * N_pad * 128 + (size_t)nst * (d / 64) * kTileKeys * 128 +
         (npass == 1 ? (size_t)N_pad * 4 : 0) + (hist ? (size_t)kScoreHistBins * 4 : 0) + sizeof(ScoreSmem);
}

cudaError_t launch_score_tc(int d, const void* K, int64_t head_stride, int H_kv, int T_len, const __nv_bfloat16* op_bf,
                            const float* op_scale, int R, KeyScale ks, float* scores, unsigned* hist,
                            WsHeader* hdr, int num_sms, cudaStream_t st) {
  if (T_len == 0) return cudaSuccess;
  const int N_pad = score_tc_pad_rows(R);
  const int npass = op_scale != nullptr ? 1 : 2;
  if (N_pad > (npass == 1 ? 512 : 256)) return cudaErrorInvalidValue;
  const bool with_hist = hist != nullptr;
  const size_t budget = 227 * 1024;
  int nst = kMaxStages;
  while (nst > 2 && score_tc_smem(d, N_pad, npass, nst, with_hist) > budget) --nst;
  const size_t smem = score_tc_smem(d, N_pad, npass, nst, with_hist);
  if (smem > budget) return cudaErrorInvalidValue;
  const int NT = npass * N_pad;
  // operand form: see ScoreMode
  const int mode = npass == 1 ? kScaled : (N_pad <= 128 ? kHiLoWide : kHiLo);
  const int tile_cols = mode == kHiLoWide ? NT : N_pad;     // accumulator columns of one tile
  const int nch = tile_cols > kUnitCols ? 2 : 1;
  const int cw = tile_cols / nch;                           // a multiple of 32
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
  launch_one<DD, MM>(grid, smem, st, kmap, omap, op_scale, T_len, N_pad, nst, nch, cw, cols, ks, scores, hist, hdr)
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
