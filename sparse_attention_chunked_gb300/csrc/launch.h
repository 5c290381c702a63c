// Internal launchers (host side) of the QUOKA kernels.  dtype: 0 = bf16,
// 1 = fp32 (quoka_dtype); d: 64 or 128.  Every launcher only enqueues on `st`
// and returns the launch status.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>
#include <utility>

namespace quoka {

// Launches `kernel` on `st` with programmatic stream serialisation, so its
// launch and prologue overlap the tail of the previous kernel (each kernel
// waits with griddepcontrol.wait before reading what that kernel wrote).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Kernels enqueued by this library in this process (read by quoka_launch_count).
extern std::atomic<unsigned long long> g_launch_count;
inline void count_launches(unsigned n) { g_launch_count.fetch_add(n, std::memory_order_relaxed); }

struct WsHeader;
// Which path launch_select_queries takes: 1 = one launch of the clustered
// kernel over whole selection rows (intermediates in shared memory only),
// 2 = mean pooling split into a clustered pass per query head that writes
// qcos and a clustered group select (when split_ok), 0 = neither fits.
int select_queries_path(int dtype, int d, const void* Q, int H_q, int G_avg, int C, int n_sel, bool split_ok);

// The N_q least similar queries per selection row.  qcos: the workspace's
// [H_q][C] floats, used by path 2.
cudaError_t launch_select_queries(int dtype, int d, const void* Q, int H_q, int G_avg, int C, int n_sel,
                                  int32_t* q_idx, float* qcos, WsHeader* hdr, cudaStream_t st,
                                  bool split_ok = true);

// Operand of the scoring stage: which rows score a KV group's keys.
//   mode 1 (per-head max pooling): the selected (head, token) pairs of the
//     group's heads; mode 0 (mean pooling): per selected token, the mean over
//     the group's heads (pre-aggregation).
//   unit: each query is normalised first (cosine score); else used as it is.
//   qmean: the rows of a head (mode 1) or of the group (mode 0) are replaced
//     by their mean (the mean over the selected tokens, folded into the
//     operand since the score is linear in the row).
struct OperandSpec {
  int mode;
  bool unit;
  bool qmean;
};

// op_f32 (CUDA-core scoring: fp32 rows [H_kv][R][d]) and op_bf (tensor-core
// scoring) may each be NULL.  op_bf rows, N_pad per pass (a multiple of 64,
// >= R):
//   op_scale == NULL: two passes, the fp32 row split into hi and lo bf16 rows,
//                     [H_kv][2][N_pad][d];
//   op_scale != NULL: mode 1 without qmean, bf16 Q only: one pass holding the
//                     selected query rows as they are, [H_kv][N_pad][d], and
//                     op_scale [H_kv][N_pad] = 1 / max(|q|, eps) (1 when not
//                     unit).
// Padding rows R..N_pad-1 of op_bf (and their scales) repeat row 0, so they
// never change a maximum.  hist (NULL or [H_kv][kScoreHistBins]) is zeroed
// for the scorer that follows.  q_idx NULL selects every position (n = C).
cudaError_t launch_build_operand(int dtype, int d, const void* Q, const int32_t* q_idx, int H_kv, int C, int G,
                                 int n, OperandSpec spec, int N_pad, float* op_f32, __nv_bfloat16* op_bf,
                                 float* op_scale, unsigned* hist, cudaStream_t st);

// How a key's score is scaled: key_norm false: 1 (dot product); else
// 1 / max(|k_t|, eps), read from k_inv[g * k_inv_stride + t] when k_inv is
// given (the key-norm cache), else computed from the key.
struct KeyScale {
  bool key_norm;
  const float* k_inv;
  int64_t k_inv_stride;
};

// The scorers can count a 12-bit histogram of their scores per KV head
// (score_bin in common.cuh: fixed-point bins for cosine scores, the top 12
// bits of order_key otherwise), where the top-B select starts.
constexpr int kScoreHistBits = 12;
constexpr int kScoreHistBins = 1 << kScoreHistBits;

// Scoring rows up to which the CUDA-core scorer takes k_score_rows (a few
// rows, each key shared by a group of lanes) instead of one key per thread.
constexpr int kScoreRowsMax = 8;

// score[g, t] = max_r (r . k_t) * scale(t).  hist, if not NULL, receives
// (adds) the histogram of score_bin(score, ks.key_norm) per head,
// [H_kv][kScoreHistBins]; launch_build_operand with the same hist zeroes it
// first.
cudaError_t launch_score_simt(int dtype, int d, const void* K, int64_t head_stride, int H_kv, int T_len,
                              const float* op_f32, int R, KeyScale ks, float* scores, unsigned* hist,
                              cudaStream_t st);

// Tensor-core scoring (bf16 keys).  op_bf / op_scale as written by
// launch_build_operand with N_pad = score_tc_pad_rows(R); npass = 1 when
// op_scale is given, else 2.
int score_tc_pad_rows(int R);
size_t score_tc_smem(int d, int N_pad, int npass, int nst, bool hist);
struct WsHeader;
cudaError_t launch_score_tc(int d, const void* K, int64_t head_stride, int H_kv, int T_len, const __nv_bfloat16* op_bf,
                            const float* op_scale, int R, KeyScale ks, float* scores, unsigned* hist,
                            WsHeader* hdr, int num_sms, cudaStream_t st);

// Raises `func`'s dynamic shared-memory limit to `bytes` on the current device (cached).
cudaError_t ensure_smem(const void* func, size_t bytes);

// TMA descriptor of a bf16 3-D tensor (see tmaps.cu).
cudaError_t make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                              uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1);

// Tensor-core attention (bf16): history rows [H_kv, n_hist, d] with head
// stride h_stride elements, then the causal chunk.
size_t attend_tc_smem(int d);
cudaError_t launch_attend_tc(int d, const void* Q, const void* Kh, const void* Vh, int64_t h_stride, int n_hist,
                             const void* Kc, const void* Vc, int H_q, int H_kv, int C, float scale, void* O,
                             float* lse, WsHeader* hdr, cudaStream_t st);

// One sequence of a ragged tensor-core attention launch: arguments as
// launch_attend_tc's (C in [1, 8192], O and lse this sequence's own).
struct AttSeq {
  const void *Q, *Kh, *Vh, *Kc, *Vc;
  int64_t h_stride;
  int n_hist, C;
  void* O;
  float* lse;
};
// Sequences per ragged launch; a longer list is covered by consecutive launches.
constexpr int kAttVarSeqs = 16;
// Every sequence's work items (query tile x head pair) in one persistent
// launch per kAttVarSeqs sequences, longest first over the whole batch.
cudaError_t launch_attend_tc_varlen(int d, const AttSeq* seqs, int nseq, int H_q, int H_kv, float scale, WsHeader* hdr,
                                    cudaStream_t st);

// The library-owned scratch of quoka_select_queries_noalloc: its device
// address on the current device (looked up on the first call per device).
constexpr size_t kNoAllocScratchBytes = 4u << 20;
cudaError_t noalloc_scratch(void** base);

// Bounded-wait self-test (see selftest.cu).
cudaError_t launch_expire_wait(WsHeader* hdr, long long limit, cudaStream_t st);

// hist: NULL, or the 12-bit histogram the scorer built for these scores
// ([H_kv][kScoreHistBins], score_bin with cosine = cosine_bins), where the
// select starts.
cudaError_t launch_topk(const float* scores, int H_kv, int T_len, int B_e, int32_t* sel, cudaStream_t st,
                        const unsigned* hist = nullptr, bool cosine_bins = false);

// Rows sel[g, j] of K and V (T_len rows per head).  An index outside
// [0, T_len) is not read: the row is written as zeros and QUOKA_ERR_DEVICE is
// recorded in hdr (when given).
cudaError_t launch_gather(int elt_bytes, int d, const void* K, const void* V, int64_t head_stride, const int32_t* sel,
                          int H_kv, int B_e, int T_len, void* Ks, void* Vs, WsHeader* hdr, cudaStream_t st);

// inv[g * inv_stride + t] = 1 / max(|K[g, t]|, eps), t in [t0, t1).
cudaError_t launch_key_inv_norms(int dtype, int d, const void* K, int64_t head_stride, int H_kv, int t0, int t1,
                                 float* inv, int64_t inv_stride, cudaStream_t st);

cudaError_t launch_append(int elt_bytes, int d, void* K, void* V, int64_t head_stride, int T_len, const void* Kc,
                          const void* Vc, int H_kv, int C, cudaStream_t st);

// Attention for chunks of at most 32 / G queries (decode), split over the
// keys: kept history rows read through sel ([H_kv][n_hist] positions; NULL =
// the first n_hist rows) straight from the cache of T_cache rows per head,
// then the causal chunk.  A position outside [0, T_cache) is not read (its
// key and value count as zero rows) and QUOKA_ERR_DEVICE is recorded in hdr.
// part: fp32 scratch of attend_decode_ws_bytes.
bool attend_decode_fits(int C, int G);
size_t attend_decode_ws_bytes(int d, int H_q, int C, int n_hist);
cudaError_t launch_attend_decode(int dtype, int d, const void* Q, const void* Kh, const void* Vh, int64_t h_stride,
                                 const int32_t* sel, int n_hist, int T_cache, const void* Kc, const void* Vc, int H_q,
                                 int H_kv, int C, float scale, void* O, float* lse, float* part, WsHeader* hdr,
                                 cudaStream_t st);

cudaError_t launch_attend_simt(int dtype, int d, const void* Q, const void* Kh, const void* Vh, int64_t h_stride,
                               int n_hist, const void* Kc, const void* Vc, int H_q, int C, int G, float scale,
                               void* O, float* lse, cudaStream_t st);

}  // namespace quoka
