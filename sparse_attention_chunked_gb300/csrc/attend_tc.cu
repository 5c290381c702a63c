// Tensor-core flash attention over [history rows ; causal chunk] (bf16, tcgen05 + TMA).
// Method: QUOKA paper summary, "Transformers and Attention" (softmax attention,
// causal mask), "Chunked prefill" (a chunk attends to the earlier keys plus
// itself, causally), "QUOKA Method" (the reduced key set feeds a dense
// attention kernel); QUOKA Explained, "MEAN and MAX do different jobs" (the
// original query heads attend).
//
// A work item is two 128-row query tiles ("slots") of two query heads of the
// same KV group over the same chunk rows, so both share every K/V tile and the
// same causal structure.  The kernel is persistent: one CTA per SM runs a
// fixed serpentine share of the longest-first item list, keeping its TMEM and
// barriers, so one item's tail (last PV, epilogue) overlaps the next item's
// Q and first K/V loads.  Keys are the history rows (selected or all) followed by
// the chunk's own rows; the history part is unmasked except past n_hist, the
// chunk part is causal.
//   S_s = Q_s K_j^T        tcgen05, A = Q (smem), B = K tile (smem), fp32 in TMEM
//   P_s = exp2(S_s - m)    softmax warpgroup of the slot, one query row per
//                          thread, written to shared memory as bf16 in the
//                          128-byte-swizzled K-major layout of an MMA operand
//   O_s += P_s V_j         tcgen05, A = P (smem), B = V tile (smem, MN-major)
// The softmax releases S_s as soon as it has loaded it, so the MMA warp
// computes S_s for block j+1 while the softmax of block j is still running;
// the running maximum is only moved (and O rescaled in TMEM) when it grows by
// more than 2^8, so most blocks never touch O.
//
// Warps (352 threads): 0 = TMA producer, 1 = TMEM owner + issuer of the S
// MMAs, 2-5 = softmax of slot 0, 6-9 = softmax of slot 1, 10 = issuer of the
// PV MMAs.  With one issuer, every wait between MMA groups (key tile, S
// released, P written, value tile) leaves the tensor pipe with only the few
// MMAs it has queued; two issuers each wait only for their own operands while
// the other keeps the pipe fed.  Every wait is bounded;
// on a timeout the CTA records QUOKA_ERR_TIMEOUT, drains what it has in
// flight, frees TMEM and exits.
#include <string.h>

#include <algorithm>

#include "launch.h"
#include "tc_common.cuh"

namespace quoka {

namespace {

constexpr int kAttThreads = 352;
constexpr int kKvStages = 3;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kPBytes = 128 * 128 * 2;   // one slot's P tile: 128 rows x 128 keys, bf16
constexpr float kRescaleThreshold = 8.0f;     // log2 units

struct AttSmem {
  uint64_t q_full;
  uint64_t q_free;       // every S MMA of the work item has completed: Q may be replaced
  uint64_t o_free[2];    // the epilogue has read O_s: the next item's first PV may overwrite it
  uint64_t kv_full[kKvStages];
  uint64_t kv_empty[kKvStages];
  uint64_t s_full[2];    // S_s of the current block is in TMEM
  uint64_t s_free[2];    // the softmax has loaded S_s (TMEM free for the next block)
  uint64_t p_full[2];    // P_s is in shared memory
  uint64_t o_done[2];    // PV_s of the current block has completed
  uint64_t drain[2];    // one per MMA issuer: its last MMAs have completed
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, WsHeader* hdr,
                                          unsigned where) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait(bar, parity, abort, hdr, where);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// 2^x on the SFU (MUFU.EX2): the hardware's approximate exponential, flushing
// subnormals; ex2(-inf) = 0.  P is rounded to bf16 afterwards.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (x0 * s + b, x1 * s + b) as one packed f32x2 FMA.
__device__ __forceinline__ void fma2(float& x0, float& x1, float s, float b) {
  unsigned long long px, ps, pb;
  asm("mov.b64 %0, {%1, %2};" : "=l"(px) : "f"(x0), "f"(x1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(ps) : "f"(s));
  asm("mov.b64 %0, {%1, %1};" : "=l"(pb) : "f"(b));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(px) : "l"(px), "l"(ps), "l"(pb));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x0), "=f"(x1) : "l"(px));
}

// (a0 + b0, a1 + b1) as one packed f32x2 add.
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  unsigned long long pa, pb;
  asm("mov.b64 %0, {%1, %2};" : "=l"(pa) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(pb) : "f"(b0), "f"(b1));
  asm("add.f32x2 %0, %1, %2;" : "=l"(pa) : "l"(pa), "l"(pb));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(pa));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// What one launch attends: NS sequences (1 for a single chunk, up to
// kAttVarSeqs for a ragged batch), each with its own tensor maps, chunk length,
// kept history rows and output.  A "run" is one query tile of one sequence;
// every run holds H_kv * pairs work items of the same length.  The items are
// dealt to the CTAs in run order.
template <int NS>
struct AttArgs {
  CUtensorMap q[NS], kh[NS], vh[NS], kc[NS], vc[NS];
  __nv_bfloat16* O[NS];
  float* lse[NS];
  int C[NS], n_hist[NS];
  int n_items;
  int n_qt;                         // NS == 1: the query tiles of the one sequence, longest (last) first
  uint16_t run[NS == 1 ? 2 : NS * 64];   // NS > 1: sequence << 8 | query tile, in work order
};

// Work item i is head pair hp of KV group g in run i / (H_kv * pairs); the
// runs of a sequence come longest (last query tile) first.  CTA c of P runs
// items c, 2P - 1 - c, 2P + c, 4P - 1 - c, ...: a serpentine over the list, so
// the CTAs that drew the longest first items draw the shortest second ones.
struct AttItem {
  int seq, qt, g, h0, n_slots, nh, n_blocks;
};

__device__ __forceinline__ int att_item_index(int c, int round, int P) {
  return (round & 1) ? (round + 1) * P - 1 - c : round * P + c;
}

template <int NS>
__device__ __forceinline__ AttItem att_item(const AttArgs<NS>& a, int i, int H_kv_pairs, int pairs, int G) {
  AttItem it;
  const int run = i / H_kv_pairs;
  if constexpr (NS == 1) {
    it.seq = 0;
    it.qt = a.n_qt - 1 - run;
  } else {
    const unsigned v = a.run[run];
    it.seq = (int)(v >> 8);
    it.qt = (int)(v & 255u);
  }
  const int rem = i - run * H_kv_pairs;
  it.g = rem / pairs;
  const int hp = rem - it.g * pairs;
  it.h0 = it.g * G + 2 * hp;
  it.n_slots = (2 * hp + 1 < G) ? 2 : 1;
  it.nh = (a.n_hist[it.seq] + 127) >> 7;
  it.n_blocks = it.nh + it.qt + 1;
  return it;
}

// One work item's softmax, rows of slot s: blocks nb .. nb + n_blocks - 1 of
// the slot's barrier phases, then the epilogue (O / l to global memory, LSE)
// and the release of O_s.  Kept out of line: inlined into the kernel's work-item
// loop its unrolled block body was scheduled about 1.4x slower.  Returns false
// once a bounded wait gave up.
template <int D>
__device__ __noinline__ bool softmax_item(AttSmem* sm, uint8_t* p_row, int s, int lane, int r, uint32_t s_addr, int nb,
                                          int n_blocks, int nh, int n_hist, int qt, int C, int h, float scale_log2,
                                          __nv_bfloat16* __restrict__ O, float* __restrict__ lse, WsHeader* hdr) {
  constexpr uint32_t kHalfBytes = 128 * 128;
  const uint32_t o_addr = s_addr + 128;
  volatile int* abort = &sm->abort;
  const int c = qt * 128 + r;                   // chunk position of the row
  bool ok = true;
  float m_used = -INFINITY, l = 0.f;           // running max of the raw logits, softmax denominator
  for (int jb = 0; jb < n_blocks; ++jb) {
    if (!(ok = warp_wait(&sm->s_full[s], (nb + jb) & 1, abort, hdr, 0x208))) break;
    tc::tc_fence_after();
    uint32_t sv[128];
    tc::tmem_ld128(s_addr, sv);
    tc::tc_fence_before();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&sm->s_free[s]);   // the MMA may now write S_s of the next block
    const bool hist = jb < nh;
    // only the last history block (if partial) and the diagonal chunk block have masked keys
    const bool need_mask = hist ? (jb == nh - 1 && (n_hist & 127) != 0) : (jb - nh == qt);
    if (need_mask) {
      // keys of this block visible to row c: [0, lim)
      const int lim = hist ? n_hist - jb * 128 : c - (jb - nh) * 128 + 1;
#pragma unroll
      for (int i2 = 0; i2 < 128; ++i2)
        if (i2 >= lim) sv[i2] = __float_as_uint(-INFINITY);
    }
    float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int i2 = 0; i2 < 64; ++i2)
      mx4[i2 & 3] = fmax3(mx4[i2 & 3], __uint_as_float(sv[2 * i2]), __uint_as_float(sv[2 * i2 + 1]));
    const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
    const float m_new = fmaxf(m_used, mx);
    const bool rescale = (m_new - m_used) * scale_log2 > kRescaleThreshold;   // true on the first block
    float alpha = 1.f;
    if (rescale) {
      alpha = ex2_approx((m_used - m_new) * scale_log2);   // 0 on the first block
      m_used = m_new;
    }
    const float neg_m = -m_used * scale_log2;
    // The probabilities are computed into registers (packed bf16, in place of the logits)
    // while PV_s of the previous block may still be reading P_s; they are stored once it is
    // done, which is also when O may be rescaled (for an item's first block the previous
    // item's epilogue already waited for it).
    float sa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i2 = 0; i2 < 128; i2 += 2) {
      float x0 = __uint_as_float(sv[i2]), x1 = __uint_as_float(sv[i2 + 1]);
      fma2(x0, x1, scale_log2, neg_m);
      const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
      if ((i2 >> 1) & 1) add2(sa[2], sa[3], p0, p1);
      else add2(sa[0], sa[1], p0, p1);
      sv[i2 >> 1] = pack_bf16x2(p0, p1);       // packed pair j lands in sv[j], below every unread logit
    }
    if (jb > 0 && !(ok = warp_wait(&sm->o_done[s], (nb + jb - 1) & 1, abort, hdr, 0x209))) break;
#pragma unroll
    for (int q = 0; q < 16; ++q) {             // 8 keys = one 16-byte chunk of P at a time
      const int hf = q >> 3, ch = q & 7;
      *reinterpret_cast<uint4*>(p_row + hf * kHalfBytes + ((ch ^ (r & 7)) << 4)) =
          make_uint4(sv[4 * q], sv[4 * q + 1], sv[4 * q + 2], sv[4 * q + 3]);
    }
    l = l * alpha + ((sa[0] + sa[1]) + (sa[2] + sa[3]));
    if (jb > 0 && __any_sync(0xffffffffu, rescale)) {   // O *= alpha in TMEM (rows without a rescale: alpha = 1)
      tc::tc_fence_after();
#pragma unroll
      for (int q4 = 0; q4 < D / 32; ++q4) {
        uint32_t ov[32];
        tc::tmem_ld32(o_addr + q4 * 32, ov);
#pragma unroll
        for (int i2 = 0; i2 < 32; ++i2) ov[i2] = __float_as_uint(__uint_as_float(ov[i2]) * alpha);
        tc::tmem_st32(o_addr + q4 * 32, ov);
      }
      tc::tmem_wait_st();
    }
    tc::fence_proxy_async_smem();              // P visible to the tensor core
    tc::tc_fence_before();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&sm->p_full[s]);
  }
  if (!ok) return false;
  // epilogue: O / l, then O_s is free for the next item's PV
  if (!warp_wait(&sm->o_done[s], (nb + n_blocks - 1) & 1, abort, hdr, 0x209)) return false;
  tc::tc_fence_after();
  const float inv = 1.f / l;
#pragma unroll
  for (int q4 = 0; q4 < D / 32; ++q4) {
    uint32_t ov[32];
    tc::tmem_ld32(o_addr + q4 * 32, ov);
    if (c < C) {
      uint4* dst = reinterpret_cast<uint4*>(O + ((size_t)h * C + c) * D + q4 * 32);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(ov[8 * v + 0]) * inv, __uint_as_float(ov[8 * v + 1]) * inv);
        w.y = pack_bf16x2(__uint_as_float(ov[8 * v + 2]) * inv, __uint_as_float(ov[8 * v + 3]) * inv);
        w.z = pack_bf16x2(__uint_as_float(ov[8 * v + 4]) * inv, __uint_as_float(ov[8 * v + 5]) * inv);
        w.w = pack_bf16x2(__uint_as_float(ov[8 * v + 6]) * inv, __uint_as_float(ov[8 * v + 7]) * inv);
        dst[v] = w;
      }
    }
  }
  tc::tc_fence_before();
  __syncwarp();
  if (lane == 0) tc::mbar_arrive(&sm->o_free[s]);
  if (lse != nullptr && c < C) lse[(size_t)h * C + c] = m_used * scale_log2 * 0.69314718055994531f + logf(l);
  return true;
}

template <int D, int NS>
__global__ void __launch_bounds__(kAttThreads, 1)
    k_attend_tc(const __grid_constant__ AttArgs<NS> a, int G, int H_kv, float scale_log2, WsHeader* hdr) {
  constexpr int HALVES = D / 64;
  constexpr uint32_t kHalfBytes = 128 * 128;            // 128 rows x 128 bytes
  constexpr uint32_t kTileBytes = HALVES * kHalfBytes;  // one Q, K or V tile of 128 rows
  constexpr uint32_t kSlotCols = 256;                   // S (128 cols) then O (D cols)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;                                  // [2][HALVES][128][128 B]
  uint8_t* p_s = q_s + 2 * kTileBytes;                  // [2][2 halves of 64 keys][128][128 B]
  uint8_t* kv_s = p_s + 2 * kPBytes;                    // [kKvStages][HALVES][128][128 B]
  AttSmem* sm = reinterpret_cast<AttSmem*>(kv_s + kKvStages * kTileBytes);

  const int pairs = (G + 1) / 2;
  const int H_kv_pairs = H_kv * pairs;
  const int n_items = a.n_items;
  const int P = gridDim.x, cta = blockIdx.x;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::mbar_init(&sm->q_full, 1);
    tc::mbar_init(&sm->q_free, 1);
    for (int s = 0; s < kKvStages; ++s) {
      tc::mbar_init(&sm->kv_full[s], 1);
      tc::mbar_init(&sm->kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&sm->s_full[s], 1);
      tc::mbar_init(&sm->s_free[s], 4);
      tc::mbar_init(&sm->p_full[s], 4);
      tc::mbar_init(&sm->o_done[s], 1);
      tc::mbar_init(&sm->o_free[s], 4);
    }
    tc::mbar_init(&sm->drain[0], 1);
    tc::mbar_init(&sm->drain[1], 1);
    sm->abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&sm->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  if (threadIdx.x == 0 && cta < n_items) {
    // The first item's query tiles do not come from the previous kernel (the
    // kept K/V rows do): start them towards L2 while that kernel finishes.
    const AttItem it0 = att_item(a, att_item_index(cta, 0, P), H_kv_pairs, pairs, G);
    const CUtensorMap* qm = &a.q[it0.seq];
    tc::tma_prefetch_desc(qm);
    for (int s = 0; s < it0.n_slots; ++s)
      for (int hf = 0; hf < HALVES; ++hf) tc::tma_prefetch_l2_3d(qm, hf * 64, it0.qt * 128, it0.h0 + s);
  }
  pdl_wait();                                   // inputs may come from the previous kernel
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile int* abort = &sm->abort;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer: per work item Q, then K_j, V_j, ...
    if (lane == 0) {
      int k = 0, n_done = 0;                    // ring items issued; work items started
      int seq_maps = -1;                         // the sequence whose maps were last prefetched
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const int i = att_item_index(cta, round, P);
        if (i >= n_items) break;
        const AttItem it = att_item(a, i, H_kv_pairs, pairs, G);
        const CUtensorMap* qm = &a.q[it.seq];
        if (it.seq != seq_maps) {
          seq_maps = it.seq;
          tc::tma_prefetch_desc(qm);
          tc::tma_prefetch_desc(&a.kc[it.seq]);
          tc::tma_prefetch_desc(&a.vc[it.seq]);
          if (it.nh > 0) {
            tc::tma_prefetch_desc(&a.kh[it.seq]);
            tc::tma_prefetch_desc(&a.vh[it.seq]);
          }
        }
        // Q of this item, once every S MMA of the previous one has read the old Q
        if (n_done > 0 && !(ok = tc::mbar_wait(&sm->q_free, (n_done - 1) & 1, abort, hdr, 0x20a))) break;
        tc::mbar_arrive_expect_tx(&sm->q_full, it.n_slots * kTileBytes);
        for (int s = 0; s < it.n_slots; ++s)
          for (int hf = 0; hf < HALVES; ++hf)
            tc::tma_load_3d(q_s + s * kTileBytes + hf * kHalfBytes, qm, &sm->q_full, hf * 64, it.qt * 128,
                            it.h0 + s);
        ++n_done;
        // the next item's query tiles towards L2, so that its Q load after this item is a short one
        const int i_next = att_item_index(cta, round + 1, P);
        if (i_next < n_items) {
          const AttItem nx = att_item(a, i_next, H_kv_pairs, pairs, G);
          const CUtensorMap* nqm = &a.q[nx.seq];
          for (int s = 0; s < nx.n_slots; ++s)
            for (int hf = 0; hf < HALVES; ++hf) tc::tma_prefetch_l2_3d(nqm, hf * 64, nx.qt * 128, nx.h0 + s);
        }
        // Ring items in the order the MMA warps consume them: K_0, then for every
        // block j: K_{j+1} (used early, by S of the next block) and V_j (used late).
        auto load = [&](int jb, int which) {    // which: 0 = K, 1 = V
          const int s = k % kKvStages;
          if (k >= kKvStages && !tc::mbar_wait(&sm->kv_empty[s], ((k / kKvStages) - 1) & 1, abort, hdr, 0x201))
            return false;
          const bool hist = jb < it.nh;
          const int row = hist ? jb * 128 : (jb - it.nh) * 128;
          const CUtensorMap* map = hist ? (which == 0 ? &a.kh[it.seq] : &a.vh[it.seq])
                                        : (which == 0 ? &a.kc[it.seq] : &a.vc[it.seq]);
          tc::mbar_arrive_expect_tx(&sm->kv_full[s], kTileBytes);
          for (int hf = 0; hf < HALVES; ++hf)
            tc::tma_load_3d(kv_s + s * kTileBytes + hf * kHalfBytes, map, &sm->kv_full[s], hf * 64, row, it.g);
          ++k;
          return true;
        };
        ok = load(0, 0);
        for (int jb = 0; ok && jb < it.n_blocks; ++jb) {
          if (jb + 1 < it.n_blocks) ok = load(jb + 1, 0);
          if (ok) ok = load(jb, 1);
        }
      }
      if (*abort) {   // let issued copies land before exiting
        if (n_done > 0) tc::mbar_drain(&sm->q_full, (n_done - 1) & 1);
        for (int kk = k - kKvStages < 0 ? 0 : k - kKvStages; kk < k; ++kk)
          tc::mbar_drain(&sm->kv_full[kk % kKvStages], (kk / kKvStages) & 1);
      }
    }
  } else if (warp == 1 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues S_s(j+1) for each slot as soon as the key tile is in and
    // the softmax has loaded S_s(j); warp 10 issues PV_s(j) as soon as the
    // value tile is in and P_s(j) is in shared memory.  Each issuer releases
    // the ring stages it read.  Block and item counts run on across work items
    // (per slot), and with them the barrier phases.
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(128, 128, false);
      constexpr uint32_t idesc_o = tc::idesc_bf16_f32(128, D, true);
      const uint32_t kvb = tc::smem_u32(kv_s), qb0 = tc::smem_u32(q_s), pb0 = tc::smem_u32(p_s);
      const bool s_issuer = warp == 1;
      bool ok = true;
      int item = 0;                              // ring item counter
      int nb[2] = {0, 0}, ni[2] = {0, 0};        // blocks / work items per slot so far
      for (int round = 0, n_done = 0; ok; ++round, ++n_done) {
        const int i = att_item_index(cta, round, P);
        if (i >= n_items) break;
        const AttItem it = att_item(a, i, H_kv_pairs, pairs, G);
        if (s_issuer) {
          auto issue_s = [&](int s, int stage) {   // S_s = Q_s K^T, K in `stage`
            const uint32_t qb = qb0 + s * kTileBytes, kb = kvb + stage * kTileBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const int hf = kk >> 2, kin = kk & 3;
              tc::mma_ss(tmem + s * kSlotCols, tc::sw128_desc(qb + hf * kHalfBytes + kin * 32, 16, 1024),
                         tc::sw128_desc(kb + hf * kHalfBytes + kin * 32, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
            }
            tc::mma_commit(&sm->s_full[s]);
          };
          if (!(ok = tc::mbar_wait(&sm->q_full, n_done & 1, abort, hdr, 0x202))) break;
          for (int jb = 0; ok && jb < it.n_blocks; ++jb) {   // key tile of block jb: ring item K_0 or K_{jb}
            const int st = item % kKvStages;
            if (!(ok = tc::mbar_wait(&sm->kv_full[st], (item / kKvStages) & 1, abort, hdr, 0x204))) break;
            for (int s = 0; s < it.n_slots; ++s) {
              const int b = nb[s] + jb;            // the slot's block count over all items
              if (b > 0 && !(ok = tc::mbar_wait(&sm->s_free[s], (b - 1) & 1, abort, hdr, 0x205))) break;
              tc::tc_fence_after();
              issue_s(s, st);
            }
            if (!ok) break;
            tc::mma_commit(&sm->kv_empty[st]);
            item += jb == 0 ? 1 : 2;             // K_0; later K_{j}, after V_{j-1} (the other issuer's)
          }
          if (!ok) break;
          item += 1;                             // the item's last V (the other issuer's)
          tc::mma_commit(&sm->q_free);           // Q no longer read once these MMAs complete
        } else {
          item += 1;                             // K_0 (the other issuer's)
          for (int jb = 0; ok && jb < it.n_blocks; ++jb) {
            if (jb + 1 < it.n_blocks) ++item;    // K_{j+1} (the other issuer's)
            const int sv = item % kKvStages;
            if (!(ok = tc::mbar_wait(&sm->kv_full[sv], (item / kKvStages) & 1, abort, hdr, 0x206))) break;
            const uint32_t vb = kvb + sv * kTileBytes;
            for (int s = 0; s < it.n_slots; ++s) {
              if (!(ok = tc::mbar_wait(&sm->p_full[s], (nb[s] + jb) & 1, abort, hdr, 0x207))) break;
              // the first PV of an item overwrites O_s: the previous item's epilogue must have read it
              if (jb == 0 && ni[s] > 0 && !(ok = tc::mbar_wait(&sm->o_free[s], (ni[s] - 1) & 1, abort, hdr, 0x20b)))
                break;
              tc::tc_fence_after();
              const uint32_t pb = pb0 + s * kPBytes;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {    // 16 keys per MMA
                const int hf = kk >> 2, kin = kk & 3;
                tc::mma_ss(tmem + s * kSlotCols + 128, tc::sw128_desc(pb + hf * kHalfBytes + kin * 32, 16, 1024),
                           tc::sw128_desc(vb + kk * 16 * 128, kHalfBytes, 1024), idesc_o,
                           (jb > 0 || kk > 0) ? 1u : 0u);
              }
              tc::mma_commit(&sm->o_done[s]);
            }
            if (!ok) break;
            tc::mma_commit(&sm->kv_empty[sv]);
            ++item;
          }
        }
        for (int s = 0; s < it.n_slots; ++s) {
          nb[s] += it.n_blocks;
          ++ni[s];
        }
      }
      uint64_t* dr = &sm->drain[s_issuer ? 0 : 1];
      tc::mma_commit(dr);                        // completes once every MMA this thread issued has finished
      tc::mbar_drain(dr, 0);
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ softmax + epilogue, one row per thread
    const int s = (warp - 2) >> 2;                 // slot
    const int quad = warp & 3;                     // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;                // row within the query tile
    const uint32_t s_addr = tmem + ((uint32_t)(quad * 32) << 16) + s * kSlotCols;
    // this row of P in the swizzled operand layout: chunk q of half h at
    // p_row + h * kHalfBytes + ((q ^ (r & 7)) << 4)
    uint8_t* p_row = p_s + s * kPBytes + (r >> 3) * 1024 + (r & 7) * 128;
    int nb = 0;                                    // blocks of this slot in earlier work items
    for (int round = 0;; ++round) {
      const int i = att_item_index(cta, round, P);
      if (i >= n_items) break;
      const AttItem it = att_item(a, i, H_kv_pairs, pairs, G);
      if (s >= it.n_slots) continue;
      if (!softmax_item<D>(sm, p_row, s, lane, r, s_addr, nb, it.n_blocks, it.nh, a.n_hist[it.seq], it.qt,
                           a.C[it.seq], it.h0 + s, scale_log2, a.O[it.seq], a.lse[it.seq], hdr))
        break;
      nb += it.n_blocks;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  pdl_launch_dependents();   // dependents launch once this CTA is done
}

}  // namespace

size_t attend_tc_smem(int d) {
  return 1024 + (size_t)(2 + kKvStages) * (d / 64) * 128 * 128 + 2 * (size_t)kPBytes + sizeof(AttSmem);
}

namespace {

// The five tensor maps of sequence slot k: Q [H_q, C, d], history K/V
// [H_kv, n_hist, d] with heads h_stride elements apart, chunk K/V [H_kv, C, d].
template <int NS>
cudaError_t fill_att_seq(AttArgs<NS>& a, int k, int d, const AttSeq& q, int H_q, int H_kv) {
  cudaError_t e;
  const uint64_t row = (uint64_t)d * 2, chunk_head = (uint64_t)q.C * d * 2;
  if ((e = make_tmap_bf16_3d(&a.q[k], q.Q, d, q.C, H_q, row, chunk_head, 64, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16_3d(&a.kc[k], q.Kc, d, q.C, H_kv, row, chunk_head, 64, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16_3d(&a.vc[k], q.Vc, d, q.C, H_kv, row, chunk_head, 64, 128)) != cudaSuccess) return e;
  if (q.n_hist > 0) {
    const uint64_t hs = (uint64_t)q.h_stride * 2;
    if ((e = make_tmap_bf16_3d(&a.kh[k], q.Kh, d, q.n_hist, H_kv, row, hs, 64, 128)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16_3d(&a.vh[k], q.Vh, d, q.n_hist, H_kv, row, hs, 64, 128)) != cudaSuccess) return e;
  } else {   // never read: no history blocks
    a.kh[k] = a.kc[k];
    a.vh[k] = a.vc[k];
  }
  a.O[k] = (__nv_bfloat16*)q.O;
  a.lse[k] = q.lse;
  a.C[k] = q.C;
  a.n_hist[k] = q.n_hist;
  return cudaSuccess;
}

template <int NS>
cudaError_t launch_att(int d, const AttArgs<NS>& a, int G, int H_kv, float scale, WsHeader* hdr, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const dim3 grid(a.n_items < sms ? a.n_items : sms);   // persistent: one CTA per SM, looping over work items
  const size_t smem = attend_tc_smem(d);
  const float scale_log2 = scale * 1.4426950408889634f;
  if (d == 64) {
    if ((e = ensure_smem((const void*)k_attend_tc<64, NS>, smem)) != cudaSuccess) return e;
    e = launch_pdl(k_attend_tc<64, NS>, grid, dim3(kAttThreads), smem, st, a, G, H_kv, scale_log2, hdr);
  } else {
    if ((e = ensure_smem((const void*)k_attend_tc<128, NS>, smem)) != cudaSuccess) return e;
    e = launch_pdl(k_attend_tc<128, NS>, grid, dim3(kAttThreads), smem, st, a, G, H_kv, scale_log2, hdr);
  }
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attend_tc(int d, const void* Q, const void* Kh, const void* Vh, int64_t h_stride, int n_hist,
                             const void* Kc, const void* Vc, int H_q, int H_kv, int C, float scale, void* O,
                             float* lse, WsHeader* hdr, cudaStream_t st) {
  AttArgs<1> a;
  memset(&a, 0, sizeof(a));
  const AttSeq q{Q, Kh, Vh, Kc, Vc, h_stride, n_hist, C, O, lse};
  cudaError_t e = fill_att_seq(a, 0, d, q, H_q, H_kv);
  if (e != cudaSuccess) return e;
  const int G = H_q / H_kv;
  a.n_qt = (C + 127) / 128;
  a.n_items = a.n_qt * H_kv * ((G + 1) / 2);
  return launch_att(d, a, G, H_kv, scale, hdr, st);
}

cudaError_t launch_attend_tc_varlen(int d, const AttSeq* seqs, int nseq, int H_q, int H_kv, float scale, WsHeader* hdr,
                                    cudaStream_t st) {
  const int G = H_q / H_kv, pairs = (G + 1) / 2;
  for (int s0 = 0; s0 < nseq; s0 += kAttVarSeqs) {
    const int n = nseq - s0 < kAttVarSeqs ? nseq - s0 : kAttVarSeqs;
    static thread_local AttArgs<kAttVarSeqs> a;   // 13 KB: kept off the stack
    memset(&a, 0, sizeof(a));
    // Runs (sequence, query tile) sequence by sequence, the sequences with the
    // longest items first and each sequence's query tiles longest (last) first.
    // The CTAs work on neighbouring items at any time, so one sequence's kept
    // and chunk K/V rows are read from HBM once and then served from L2 (a
    // batch-wide longest-first order interleaves every sequence's runs, and
    // the rows are evicted between one query tile and the next).
    int order[kAttVarSeqs], longest[kAttVarSeqs];
    for (int k = 0; k < n; ++k) {
      const AttSeq& q = seqs[s0 + k];
      if (q.C < 1 || q.C > 64 * 128 || q.n_hist < 0) return cudaErrorInvalidValue;
      cudaError_t e = fill_att_seq(a, k, d, q, H_q, H_kv);
      if (e != cudaSuccess) return e;
      order[k] = k;
      longest[k] = (q.n_hist + 127) / 128 + (q.C + 127) / 128;
    }
    std::stable_sort(order, order + n, [&](int x, int y) { return longest[x] > longest[y]; });
    int n_runs = 0;
    for (int o = 0; o < n; ++o) {
      const int k = order[o];
      for (int qt = (seqs[s0 + k].C + 127) / 128 - 1; qt >= 0; --qt) a.run[n_runs++] = (uint16_t)((k << 8) | qt);
    }
    a.n_items = n_runs * H_kv * pairs;
    cudaError_t e = launch_att(d, a, G, H_kv, scale, hdr, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace quoka
