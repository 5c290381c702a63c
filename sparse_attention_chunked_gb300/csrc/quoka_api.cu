// C ABI of libquoka.so: argument checks, workspace layout and the launch
// sequence of each entry point.  Declarations and their contracts are in
// include/quoka.h.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "quoka.h"
#include "common.cuh"
#include "launch.h"

namespace {

using namespace quoka;

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int elt_bytes(int dtype) { return dtype == QUOKA_DTYPE_FP32 ? 4 : 2; }

int64_t head_stride(const quoka_shape* s) {
  return s->kv_head_stride ? s->kv_head_stride : (int64_t)s->T * s->d;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int check_shape(const quoka_shape* s) {
  if (s == nullptr) return QUOKA_ERR_INVALID_ARG;
  if (s->H_q < 1 || s->H_kv < 1 || s->H_q % s->H_kv != 0) return QUOKA_ERR_INVALID_ARG;
  if (s->C < 1 || s->T < 0) return QUOKA_ERR_INVALID_ARG;
  if (s->dtype != QUOKA_DTYPE_BF16 && s->dtype != QUOKA_DTYPE_FP32) return QUOKA_ERR_INVALID_ARG;
  if (s->kv_head_stride < 0 || head_stride(s) < (int64_t)s->T * s->d) return QUOKA_ERR_INVALID_ARG;
  if (s->d != 64 && s->d != 128) return QUOKA_ERR_UNSUPPORTED;
  if (s->C > 8192) return QUOKA_ERR_UNSUPPORTED;
  if ((head_stride(s) * elt_bytes(s->dtype)) % 16 != 0) return QUOKA_ERR_ALIGNMENT;
  return QUOKA_OK;
}

struct Params {
  int gqa;        // quoka_gqa_pool
  int engine;     // quoka_engine
  float scale;
  bool dot;       // QUOKA_FLAG_SCORE_DOT
  bool qmean;     // QUOKA_FLAG_QUERY_MEAN
};

int read_params(const quoka_params* p, const quoka_shape* s, Params* out) {
  out->gqa = QUOKA_GQA_MEAN_PREAGG;
  out->engine = QUOKA_ENGINE_AUTO;
  out->scale = 1.0f / sqrtf((float)s->d);
  out->dot = out->qmean = false;
  if (p == nullptr) return QUOKA_OK;
  if (p->gqa_pool != QUOKA_GQA_MEAN_PREAGG && p->gqa_pool != QUOKA_GQA_MAX) return QUOKA_ERR_INVALID_ARG;
  if (p->engine < QUOKA_ENGINE_AUTO || p->engine > QUOKA_ENGINE_TENSOR) return QUOKA_ERR_INVALID_ARG;
  if ((p->flags & ~(QUOKA_FLAG_SCORE_DOT | QUOKA_FLAG_QUERY_MEAN)) != 0) return QUOKA_ERR_INVALID_ARG;
  out->dot = (p->flags & QUOKA_FLAG_SCORE_DOT) != 0;
  out->qmean = (p->flags & QUOKA_FLAG_QUERY_MEAN) != 0;
  if (!(p->softmax_scale == p->softmax_scale)) return QUOKA_ERR_INVALID_ARG;   // NaN
  out->gqa = p->gqa_pool;
  out->engine = p->engine;
  if (p->softmax_scale > 0.f) out->scale = p->softmax_scale;
  return QUOKA_OK;
}

int n_sel_of(const quoka_shape* s, int N_q) { return N_q < s->C ? N_q : s->C; }

// Scoring rows per KV group: every selected (head, token) for per-head max
// pooling, one pre-aggregated row per token for mean pooling; the mean over
// the selected tokens is linear, so QUOKA_FLAG_QUERY_MEAN folds the tokens
// into one row per head (max pooling) or per group (mean pooling).
int score_rows(const quoka_shape* s, int N_q, const Params& p) {
  const int n = n_sel_of(s, N_q), G = s->H_q / s->H_kv;
  if (p.gqa == QUOKA_GQA_MAX) return p.qmean ? G : G * n;
  return p.qmean ? 1 : n;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 148;
  return n;
}

// Operand rows per scoring row of the tensor-core scorer: 2 = hi + lo bf16
// rows, 1 = the raw bf16 query rows with an fp32 scale per row applied in the
// epilogue.  Rows that are averages (mean pooling, or the mean over tokens)
// have no exact bf16 form and go in as hi + lo; per-head max pooling scores
// with the query rows themselves (one MMA pass, half the tensor work).
int score_npass(const quoka_shape* s, int N_pad, const Params& p) {
  (void)s;
  (void)N_pad;
  return (p.gqa == QUOKA_GQA_MAX && !p.qmean) ? 1 : 2;
}

// Whether the scoring stage can run on the tensor cores: bf16 keys, at most
// 512 scaled rows or 256 hi/lo rows, and an operand that fits shared memory
// next to two key stages and the 12-bit score histogram.
bool score_tc_fits(const quoka_shape* s, int N_q, const Params& p) {
  if (s->dtype != QUOKA_DTYPE_BF16) return false;
  const int N_pad = score_tc_pad_rows(score_rows(s, N_q, p));
  const int npass = score_npass(s, N_pad, p);
  return N_pad <= (npass == 1 ? 512 : 256) && score_tc_smem(s->d, N_pad, npass, 2, true) <= 227 * 1024;
}

// Chunks of at most 32 / G queries (decode) attend through the split-key
// CUDA-core kernel unless the tensor-core engine is forced.
bool use_decode(const Params& p, const quoka_shape* s) {
  return p.engine != QUOKA_ENGINE_TENSOR && attend_decode_fits(s->C, s->H_q / s->H_kv);
}

// Which kernels run (stage 0 = scoring, 1 = attention).  Tensor-core kernels are bf16 only.
bool use_tensor_cores(const Params& p, const quoka_shape* s, int stage, int N_q = 1) {
  if (p.engine == QUOKA_ENGINE_SIMT || s->dtype != QUOKA_DTYPE_BF16) return false;
  if (stage == 0) return score_tc_fits(s, N_q, p);
  return !use_decode(p, s) && attend_tc_smem(s->d) <= 227 * 1024;
}

// Workspace regions, in order; each stage only touches the prefix it needs:
//   [header][select scratch][score scratch][chunk intermediates]
struct Layout {
  size_t qcos, select_end;
  size_t op_f32, op_bf, op_scale, score_end;
  size_t q_idx, scores, hist, sel, ksel, vsel, dec, total;
};

// Regions start at `start` (just past the header for a single call; a lane's
// slice for the ragged entry point).  The header is always the workspace's
// first 256 bytes, shared by every lane.  gather = false leaves out the
// gathered K/V rows (the ragged entry point keeps them outside the lanes).
Layout make_layout(const quoka_shape* s, int N_q, int B, const Params& p, size_t start = sizeof(WsHeader),
                   bool gather = true) {
  Layout L;
  const size_t H_q = s->H_q, H_kv = s->H_kv, C = s->C, d = s->d, T = s->T;
  size_t o = start;
  L.qcos = o;   o = align_up(o + H_q * C * 4);   // per-head cosines of the split mean-pooling select
  L.select_end = o;
  const size_t R = (size_t)score_rows(s, N_q > 0 ? N_q : 1, p);
  const size_t N_pad = (size_t)score_tc_pad_rows((int)R);
  L.op_f32 = o;   o = align_up(o + H_kv * R * d * 4);
  L.op_bf = o;    o = align_up(o + H_kv * (size_t)score_npass(s, (int)N_pad, p) * N_pad * d * 2);
  L.op_scale = o; o = align_up(o + H_kv * N_pad * 4);
  L.score_end = o;
  const size_t n = (size_t)n_sel_of(s, N_q > 0 ? N_q : 1);
  const size_t B_e = (size_t)(B < s->T ? B : s->T);
  L.q_idx = o;  o = align_up(o + H_q * n * 4);
  L.scores = o; o = align_up(o + H_kv * T * 4);
  L.hist = o;   o = align_up(o + H_kv * kScoreHistBins * 4);
  L.sel = o;    o = align_up(o + H_kv * B_e * 4);
  const size_t kept = gather ? H_kv * B_e * d * elt_bytes(s->dtype) : 0;
  L.ksel = o;   o = align_up(o + kept);
  L.vsel = o;   o = align_up(o + kept);
  L.dec = o;    o = align_up(o + (use_decode(p, s) ? attend_decode_ws_bytes(s->d, s->H_q, s->C, s->T) : 0));
  L.total = o;
  return L;
}

int check_ws(const void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr || ((uintptr_t)ws % kAlign) != 0 || ws_bytes < need) return QUOKA_ERR_WORKSPACE;
  return QUOKA_OK;
}

thread_local cudaError_t t_last_cuda_error = cudaSuccess;

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return QUOKA_OK;
  t_last_cuda_error = e;
  return QUOKA_ERR_CUDA;
}

template <typename P> P* at(void* ws, size_t off) { return reinterpret_cast<P*>(static_cast<char*>(ws) + off); }

#define QUOKA_TRY(x)                 \
  do {                               \
    int _rc = (x);                   \
    if (_rc != QUOKA_OK) return _rc; \
  } while (0)

#define QUOKA_CUDA(x) QUOKA_TRY(cuda_status(x))

int run_select(const quoka_shape* s, const void* Q, int n, const Params& p, int32_t* q_idx, void* ws,
               const Layout& L, cudaStream_t st, bool split_ok = true) {
  const int G = s->H_q / s->H_kv;
  const int G_avg = p.gqa == QUOKA_GQA_MAX ? 1 : G;
  // N_q >= C keeps every query (a decode step's one token, say): the ascending
  // positions 0..C-1, with no cosines to compute
  if (n >= s->C) return cuda_status(launch_topk(nullptr, s->H_q / G_avg, s->C, s->C, q_idx, st));
  if (select_queries_path(s->dtype, s->d, Q, s->H_q, G_avg, s->C, n, split_ok) == 0) return QUOKA_ERR_UNSUPPORTED;
  return cuda_status(launch_select_queries(s->dtype, s->d, Q, s->H_q, G_avg, s->C, n, q_idx, at<float>(ws, L.qcos),
                                           at<WsHeader>(ws, 0), st, split_ok));
}

// An optional cache of 1 / max(|k_t|, eps) for the history keys ([H_kv] rows
// `stride` apart), written when the keys were appended.
struct KeyCache {
  const float* inv = nullptr;
  int64_t stride = 0;
};

int run_score(const quoka_shape* s, const void* Q, const int32_t* q_idx, int n, const void* K_hist,
              const Params& p, float* scores, void* ws, const Layout& L, cudaStream_t st, KeyCache kc = KeyCache(),
              unsigned* hist = nullptr) {
  const int G = s->H_q / s->H_kv;
  OperandSpec os;
  os.mode = p.gqa == QUOKA_GQA_MAX ? 1 : 0;
  os.unit = !p.dot;
  os.qmean = p.qmean;
  const int R = score_rows(s, n, p);
  const int N_pad = score_tc_pad_rows(R);
  const bool tc = use_tensor_cores(p, s, 0, n);
  if (p.engine == QUOKA_ENGINE_TENSOR && !tc) return QUOKA_ERR_UNSUPPORTED;
  float* op_scale = tc && score_npass(s, N_pad, p) == 1 ? at<float>(ws, L.op_scale) : nullptr;
  QUOKA_CUDA(launch_build_operand(s->dtype, s->d, Q, q_idx, s->H_kv, s->C, G, n, os, N_pad,
                                  tc ? nullptr : at<float>(ws, L.op_f32), tc ? at<__nv_bfloat16>(ws, L.op_bf) : nullptr,
                                  op_scale, hist, st));
  const KeyScale ks{!p.dot, kc.inv, kc.stride};
  if (tc)
    return cuda_status(launch_score_tc(s->d, K_hist, head_stride(s), s->H_kv, s->T, at<__nv_bfloat16>(ws, L.op_bf),
                                       op_scale, R, ks, scores, hist, at<WsHeader>(ws, 0), num_sms(), st));
  return cuda_status(launch_score_simt(s->dtype, s->d, K_hist, head_stride(s), s->H_kv, s->T,
                                       at<float>(ws, L.op_f32), R, ks, scores, hist, st));
}

// Attention over n_hist history rows (rows sel[g][0..n_hist) of Kh/Vh, or the
// first n_hist when sel is NULL) plus the causal chunk.  The tensor-core and
// prefill CUDA-core kernels take the rows contiguous (sel must be NULL); the
// decode kernel reads them through sel and uses the scratch at ws + dec_off.
int run_attend(const quoka_shape* s, const void* Q, const void* Kh, const void* Vh, int64_t h_stride,
               const int32_t* sel, int n_hist, const void* Kc, const void* Vc, const Params& p, void* O, float* lse,
               void* ws, size_t dec_off, cudaStream_t st) {
  const int G = s->H_q / s->H_kv;
  if (use_decode(p, s))   // rows read through sel come from a cache of T rows, else Kh holds n_hist rows
    return cuda_status(launch_attend_decode(s->dtype, s->d, Q, Kh, Vh, h_stride, sel, n_hist,
                                            sel != nullptr ? s->T : n_hist, Kc, Vc, s->H_q, s->H_kv, s->C, p.scale, O,
                                            lse, at<float>(ws, dec_off), at<WsHeader>(ws, 0), st));
  if (sel != nullptr) return QUOKA_ERR_DEVICE;   // not reached: only the decode kernel reads through sel
  const bool tc = use_tensor_cores(p, s, 1);
  if (p.engine == QUOKA_ENGINE_TENSOR && !tc) return QUOKA_ERR_UNSUPPORTED;
  if (tc)
    return cuda_status(launch_attend_tc(s->d, Q, Kh, Vh, h_stride, n_hist, Kc, Vc, s->H_q, s->H_kv, s->C, p.scale, O,
                                        lse, at<WsHeader>(ws, 0), st));
  return cuda_status(launch_attend_simt(s->dtype, s->d, Q, Kh, Vh, h_stride, n_hist, Kc, Vc, s->H_q, s->C, G,
                                        p.scale, O, lse, st));
}

bool aligned4(const void* p) { return ((uintptr_t)p & 3u) == 0; }

// The key-norm cache: a 4-byte aligned fp32 array with rows of at least
// `len` entries, one row per KV head.
int check_norm_cache(const quoka_shape* s, const float* inv, int64_t stride, int64_t len) {
  if (inv == nullptr || stride < len || stride < 1) return QUOKA_ERR_INVALID_ARG;
  if (((uintptr_t)inv & 3u) != 0) return QUOKA_ERR_ALIGNMENT;
  (void)s;
  return QUOKA_OK;
}

// Pointer checks shared by quoka_chunk_attend and each sequence of the ragged
// entry point.  lse and sel_out are written one element at a time and need
// only 4-byte alignment.
int check_chunk_args(const quoka_shape* shape, const void* Q, const void* K_hist, const void* V_hist,
                     const void* K_chunk, const void* V_chunk, int N_q, int B, const void* O, const float* lse,
                     const int32_t* sel_out) {
  if (N_q < 1 || B < 1 || Q == nullptr || K_chunk == nullptr || V_chunk == nullptr || O == nullptr)
    return QUOKA_ERR_INVALID_ARG;
  if (shape->T > 0 && (K_hist == nullptr || V_hist == nullptr)) return QUOKA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K_hist) || !aligned16(V_hist) || !aligned16(K_chunk) || !aligned16(V_chunk) ||
      !aligned16(O) || !aligned4(lse) || !aligned4(sel_out))
    return QUOKA_ERR_ALIGNMENT;
  return QUOKA_OK;
}

// Where the ragged entry point wants a chunk's kept K/V rows ([H_kv, B, d]
// each): that chunk's attention runs later, in one launch over the batch.
struct KeepOnly {
  void* K;
  void* V;
};

// One chunk, arguments already checked: select queries, score the history,
// keep the top-B keys, gather them and attend.  T = 0 or B >= T attends to the
// whole history instead.  With `keep`, the chunk stops after the gather (into
// keep's rows; nothing to gather when every history key is kept).
int run_chunk(const quoka_shape* shape, const void* Q, const void* K_hist, const void* V_hist, const void* K_chunk,
              const void* V_chunk, int N_q, int B, const Params& p, void* O, float* lse, int32_t* sel_out, void* ws,
              const Layout& L, cudaStream_t st, KeyCache kc = KeyCache(), const KeepOnly* keep = nullptr) {
  const int T = shape->T;
  if (T == 0 || B >= T) {   // every history key is kept: dense chunked-prefill attention
    if (sel_out != nullptr && T > 0) QUOKA_CUDA(launch_topk(nullptr, shape->H_kv, T, T, sel_out, st));
    if (keep != nullptr) return QUOKA_OK;
    return run_attend(shape, Q, K_hist, V_hist, head_stride(shape), nullptr, T, K_chunk, V_chunk, p, O, lse, ws,
                      L.dec, st);
  }
  const int n = n_sel_of(shape, N_q);
  int32_t* q_idx = at<int32_t>(ws, L.q_idx);
  float* scores = at<float>(ws, L.scores);
  int32_t* sel = sel_out != nullptr ? sel_out : at<int32_t>(ws, L.sel);
  // N_q >= C keeps every query (a decode step): the operand kernel takes them
  // all directly, with no index list to write first
  const bool all_queries = n >= shape->C;
  if (!all_queries) QUOKA_TRY(run_select(shape, Q, n, p, q_idx, ws, L, st));
  // the scorer also counts a 12-bit histogram of its scores (fixed-point bins
  // for cosines), where the top-B select then starts
  unsigned* hist = at<unsigned>(ws, L.hist);
  QUOKA_TRY(run_score(shape, Q, all_queries ? nullptr : q_idx, n, K_hist, p, scores, ws, L, st, kc, hist));
  QUOKA_CUDA(launch_topk(scores, shape->H_kv, T, B, sel, st, hist, !p.dot));
  if (use_decode(p, shape))   // the decode kernel reads the kept rows through sel: no gathered copy
    return run_attend(shape, Q, K_hist, V_hist, head_stride(shape), sel, B, K_chunk, V_chunk, p, O, lse, ws, L.dec,
                      st);
  void* ksel = keep != nullptr ? keep->K : at<void>(ws, L.ksel);
  void* vsel = keep != nullptr ? keep->V : at<void>(ws, L.vsel);
  QUOKA_CUDA(launch_gather(elt_bytes(shape->dtype), shape->d, K_hist, V_hist, head_stride(shape), sel, shape->H_kv, B,
                           T, ksel, vsel, at<WsHeader>(ws, 0), st));
  if (keep != nullptr) return QUOKA_OK;
  return run_attend(shape, Q, ksel, vsel, (int64_t)B * shape->d, nullptr, B, K_chunk, V_chunk, p, O, lse, ws, L.dec,
                    st);
}

// Ragged batch: the prefix sums must start at 0, never decrease, and give
// every sequence C_s <= 8192 and T_s < 2^31.
int check_varlen(const quoka_varlen_shape* v, const int64_t* cu_T, const int64_t* cu_C) {
  if (v == nullptr || cu_T == nullptr || cu_C == nullptr) return QUOKA_ERR_INVALID_ARG;
  if (v->nseq < 1 || v->reserved != 0 || cu_T[0] != 0 || cu_C[0] != 0) return QUOKA_ERR_INVALID_ARG;
  for (int s = 0; s < v->nseq; ++s) {
    const int64_t C = cu_C[s + 1] - cu_C[s], T = cu_T[s + 1] - cu_T[s];
    if (C < 0 || T < 0) return QUOKA_ERR_INVALID_ARG;
    if (C > 8192 || T > INT32_MAX) return QUOKA_ERR_UNSUPPORTED;
  }
  const quoka_shape first = {0, v->H_q, v->H_kv, 1, 0, v->d, v->dtype};
  return check_shape(&first);   // the head layout, d and dtype
}

quoka_shape seq_shape(const quoka_varlen_shape* v, const int64_t* cu_T, const int64_t* cu_C, int s) {
  quoka_shape sh;
  sh.kv_head_stride = 0;
  sh.H_q = v->H_q;
  sh.H_kv = v->H_kv;
  sh.C = (int32_t)(cu_C[s + 1] - cu_C[s]);
  sh.T = (int32_t)(cu_T[s + 1] - cu_T[s]);
  sh.d = v->d;
  sh.dtype = v->dtype;
  return sh;
}

struct SeqArgs {
  quoka_shape shape;
  const void *Q, *K_hist, *V_hist, *K_chunk, *V_chunk;
  void* O;
  float* lse;
  int32_t* sel_out;
  Params p;
  Layout L;
  bool joint;        // attends in the batch's joint tensor-core launch
  size_t kept;       // joint and selecting: offset of its gathered K rows (V rows follow)
  double work;
};

// A ragged batch's sequences whose attention runs on the tensor cores (bf16,
// more than decode size) attend in one joint launch over the whole batch, so
// that its work items balance across the SMs; the lanes run their selection
// only.  The rest (decode-size chunks, fp32) run whole on the lanes.
bool joint_attention(const quoka_shape& sh, const Params& p) { return use_tensor_cores(p, &sh, 1); }

// Bytes of one joint sequence's gathered K and V rows (both), 0 when it keeps
// every history key (attended in place) or has none.
size_t joint_kept_bytes(const quoka_shape& sh, int B) {
  if (sh.T == 0 || B >= sh.T) return 0;
  return 2 * align_up((size_t)sh.H_kv * B * sh.d * elt_bytes(sh.dtype));
}

// Streams the ragged entry point runs sequences on: sequences of one batch
// share nothing, so their launches may overlap on the GPU.
constexpr int kMaxLanes = 8;

int varlen_lanes(const quoka_varlen_shape* v, const int64_t* cu_C) {
  int busy = 0;
  for (int s = 0; s < v->nseq; ++s) busy += cu_C[s + 1] > cu_C[s];
  return std::max(1, std::min(busy, kMaxLanes));
}

// Workspace of one lane: room for the largest sequence's regions (without
// the gathered rows of joint sequences); *kept: the joint sequences' gathered
// rows, which sit between the header and the lanes.
int varlen_lane_bytes(const quoka_varlen_shape* v, const int64_t* cu_T, const int64_t* cu_C, int N_q, int B,
                      const quoka_params* params, size_t* out, size_t* kept) {
  size_t lane = 0, rows = 0;
  for (int s = 0; s < v->nseq; ++s) {
    const quoka_shape sh = seq_shape(v, cu_T, cu_C, s);
    if (sh.C == 0) continue;
    Params p;
    QUOKA_TRY(read_params(params, &sh, &p));
    const bool joint = joint_attention(sh, p);
    lane = std::max(lane, make_layout(&sh, N_q, B, p, sizeof(WsHeader), !joint).total - sizeof(WsHeader));
    if (joint) rows += joint_kept_bytes(sh, B);
  }
  *out = align_up(lane);
  *kept = rows;
  return QUOKA_OK;
}

// Relative cost of a sequence, for balancing lanes: the history it scores and
// (unless it attends in the joint launch) the keys each query attends to.
double seq_work(const quoka_shape& s, int B, bool attends) {
  const double Be = std::min(B, s.T);
  return (double)s.H_kv * s.T * s.d * 2.0 / 8.0 +
         (attends ? (double)s.H_q * s.C * (Be + 0.5 * s.C) * s.d * 4.0 / 1000.0 : 0.0);
}

struct LaneStreams {
  std::mutex mu;
  cudaStream_t stream[kMaxLanes - 1];
  cudaEvent_t fork, join[kMaxLanes - 1];
};

// Per device, created on first use and kept for the life of the process.
cudaError_t lane_streams(LaneStreams** out) {
  static std::mutex mu;
  static LaneStreams* per_dev[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> guard(mu);
  if (per_dev[dev] == nullptr) {
    LaneStreams* ls = new LaneStreams();
    if ((e = cudaEventCreateWithFlags(&ls->fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    for (int l = 0; l < kMaxLanes - 1; ++l) {
      if ((e = cudaStreamCreateWithFlags(&ls->stream[l], cudaStreamNonBlocking)) != cudaSuccess) return e;
      if ((e = cudaEventCreateWithFlags(&ls->join[l], cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    per_dev[dev] = ls;
  }
  *out = per_dev[dev];
  return cudaSuccess;
}

}  // namespace

namespace quoka {
std::atomic<unsigned long long> g_launch_count{0};
}

extern "C" {

int quoka_stage_engine(const quoka_shape* shape, const quoka_params* params, int stage) {
  const int rc = check_shape(shape);
  if (rc != QUOKA_OK) return -rc;
  Params p;
  const int rp = read_params(params, shape, &p);
  if (rp != QUOKA_OK) return -rp;
  if (stage != 0 && stage != 1) return -QUOKA_ERR_INVALID_ARG;
  return use_tensor_cores(p, shape, stage, 1) ? QUOKA_ENGINE_TENSOR : QUOKA_ENGINE_SIMT;
}

const char* quoka_last_cuda_error_string(void) { return cudaGetErrorString(t_last_cuda_error); }

uint64_t quoka_launch_count(void) { return quoka::g_launch_count.load(std::memory_order_relaxed); }

const char* quoka_status_string(int status) {
  switch (status) {
    case QUOKA_OK: return "QUOKA_OK";
    case QUOKA_ERR_INVALID_ARG: return "QUOKA_ERR_INVALID_ARG";
    case QUOKA_ERR_UNSUPPORTED: return "QUOKA_ERR_UNSUPPORTED";
    case QUOKA_ERR_WORKSPACE: return "QUOKA_ERR_WORKSPACE";
    case QUOKA_ERR_ALIGNMENT: return "QUOKA_ERR_ALIGNMENT";
    case QUOKA_ERR_CUDA: return "QUOKA_ERR_CUDA";
    case QUOKA_ERR_TIMEOUT: return "QUOKA_ERR_TIMEOUT";
    case QUOKA_ERR_DEVICE: return "QUOKA_ERR_DEVICE";
    default: return "QUOKA_ERR_UNKNOWN";
  }
}

int quoka_workspace_size(const quoka_shape* shape, int N_q, int B, const quoka_params* params, size_t* bytes) {
  QUOKA_TRY(check_shape(shape));
  Params p;
  QUOKA_TRY(read_params(params, shape, &p));
  if (N_q < 1 || B < 1 || bytes == nullptr) return QUOKA_ERR_INVALID_ARG;
  *bytes = make_layout(shape, N_q, B, p).total;
  return QUOKA_OK;
}

int quoka_select_queries(const quoka_shape* shape, const void* Q, int N_q, const quoka_params* params,
                         int32_t* q_idx, void* ws, size_t ws_bytes, void* stream) {
  QUOKA_TRY(check_shape(shape));
  Params p;
  QUOKA_TRY(read_params(params, shape, &p));
  if (N_q < 1 || Q == nullptr || q_idx == nullptr) return QUOKA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(q_idx)) return QUOKA_ERR_ALIGNMENT;
  const Layout L = make_layout(shape, N_q, 1, p);
  QUOKA_TRY(check_ws(ws, ws_bytes, L.select_end));
  return run_select(shape, Q, n_sel_of(shape, N_q), p, q_idx, ws, L, (cudaStream_t)stream);
}

int quoka_select_queries_noalloc(const quoka_shape* shape, const void* Q, int N_q, const quoka_params* params,
                                 int32_t* q_idx, void* stream) {
  QUOKA_TRY(check_shape(shape));
  Params p;
  QUOKA_TRY(read_params(params, shape, &p));
  if (N_q < 1 || Q == nullptr || q_idx == nullptr) return QUOKA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(q_idx)) return QUOKA_ERR_ALIGNMENT;
  // The library's scratch array stands in for the workspace, laid out the same
  // way (error header first).  Only the split of mean pooling reads and writes
  // the region after the header (the per-head cosines), and only when the
  // layout fits the array; otherwise mean pooling runs the one-launch kernel
  // over whole groups where its shared memory allows.
  const Layout L = make_layout(shape, N_q, 1, p);
  const int n = n_sel_of(shape, N_q);
  const int G_avg = p.gqa == QUOKA_GQA_MAX ? 1 : shape->H_q / shape->H_kv;
  const bool fits = L.select_end <= kNoAllocScratchBytes;
  if (n < shape->C && select_queries_path(shape->dtype, shape->d, Q, shape->H_q, G_avg, shape->C, n, fits) == 0)
    return QUOKA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  QUOKA_CUDA(noalloc_scratch(&scratch));
  return run_select(shape, Q, n, p, q_idx, scratch, L, (cudaStream_t)stream, fits);
}

int quoka_score_keys(const quoka_shape* shape, const void* Q, const int32_t* q_idx, int N_q, const void* K_hist,
                     const quoka_params* params, float* scores, void* ws, size_t ws_bytes, void* stream) {
  QUOKA_TRY(check_shape(shape));
  Params p;
  QUOKA_TRY(read_params(params, shape, &p));
  if (N_q < 1 || Q == nullptr || q_idx == nullptr || K_hist == nullptr || scores == nullptr)
    return QUOKA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(q_idx) || !aligned16(K_hist) || !aligned16(scores)) return QUOKA_ERR_ALIGNMENT;
  const Layout L = make_layout(shape, N_q, 1, p);
  QUOKA_TRY(check_ws(ws, ws_bytes, L.score_end));
  if (shape->T == 0) return QUOKA_OK;
  return run_score(shape, Q, q_idx, n_sel_of(shape, N_q), K_hist, p, scores, ws, L, (cudaStream_t)stream);
}

int quoka_score_keys_cached(const quoka_shape* shape, const void* Q, const int32_t* q_idx, int N_q,
                            const void* K_hist, const float* k_inv_norm, int64_t norm_head_stride,
                            const quoka_params* params, float* scores, void* ws, size_t ws_bytes, void* stream) {
  QUOKA_TRY(check_shape(shape));
  Params p;
  QUOKA_TRY(read_params(params, shape, &p));
  QUOKA_TRY(check_norm_cache(shape, k_inv_norm, norm_head_stride, shape->T));
  if (N_q < 1 || Q == nullptr || q_idx == nullptr || K_hist == nullptr || scores == nullptr)
    return QUOKA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(q_idx) || !aligned16(K_hist) || !aligned16(scores)) return QUOKA_ERR_ALIGNMENT;
  const Layout L = make_layout(shape, N_q, 1, p);
  QUOKA_TRY(check_ws(ws, ws_bytes, L.score_end));
  if (shape->T == 0) return QUOKA_OK;
  KeyCache kc;
  kc.inv = k_inv_norm;
  kc.stride = norm_head_stride;
  return run_score(shape, Q, q_idx, n_sel_of(shape, N_q), K_hist, p, scores, ws, L, (cudaStream_t)stream, kc);
}

int quoka_key_inv_norms(const quoka_shape* shape, const void* K_hist, int t0, int t1, float* k_inv_norm,
                        int64_t norm_head_stride, void* stream) {
  QUOKA_TRY(check_shape(shape));
  if (K_hist == nullptr || t0 < 0 || t1 < t0 || t1 > shape->T) return QUOKA_ERR_INVALID_ARG;
  QUOKA_TRY(check_norm_cache(shape, k_inv_norm, norm_head_stride, t1));
  if (!aligned16(K_hist)) return QUOKA_ERR_ALIGNMENT;
  return cuda_status(launch_key_inv_norms(shape->dtype, shape->d, K_hist, head_stride(shape), shape->H_kv, t0, t1,
                                          k_inv_norm, norm_head_stride, (cudaStream_t)stream));
}

int quoka_topk(const quoka_shape* shape, const float* scores, int B, int32_t* sel, void* ws, size_t ws_bytes,
               void* stream) {
  QUOKA_TRY(check_shape(shape));
  if (B < 1 || scores == nullptr || sel == nullptr) return QUOKA_ERR_INVALID_ARG;
  if (!aligned16(scores) || !aligned16(sel)) return QUOKA_ERR_ALIGNMENT;
  QUOKA_TRY(check_ws(ws, ws_bytes, sizeof(WsHeader)));
  const int B_e = B < shape->T ? B : shape->T;
  return cuda_status(launch_topk(scores, shape->H_kv, shape->T, B_e, sel, (cudaStream_t)stream));
}

int quoka_gather(const quoka_shape* shape, const void* K_hist, const void* V_hist, const int32_t* sel, int B_e,
                 void* K_sel, void* V_sel, void* stream) {
  QUOKA_TRY(check_shape(shape));
  if (B_e < 0 || B_e > shape->T) return QUOKA_ERR_INVALID_ARG;
  if (B_e == 0) return QUOKA_OK;
  if (!K_hist || !V_hist || !sel || !K_sel || !V_sel) return QUOKA_ERR_INVALID_ARG;
  if (!aligned16(K_hist) || !aligned16(V_hist) || !aligned16(sel) || !aligned16(K_sel) || !aligned16(V_sel))
    return QUOKA_ERR_ALIGNMENT;
  return cuda_status(launch_gather(elt_bytes(shape->dtype), shape->d, K_hist, V_hist, head_stride(shape), sel,
                                   shape->H_kv, B_e, shape->T, K_sel, V_sel, nullptr, (cudaStream_t)stream));
}

int quoka_sparse_attend(const quoka_shape* shape, const void* Q, const void* K_sel, const void* V_sel, int B_e,
                        const void* K_chunk, const void* V_chunk, const quoka_params* params, void* O, float* lse,
                        void* ws, size_t ws_bytes, void* stream) {
  QUOKA_TRY(check_shape(shape));
  Params p;
  QUOKA_TRY(read_params(params, shape, &p));
  if (B_e < 0 || Q == nullptr || K_chunk == nullptr || V_chunk == nullptr || O == nullptr) return QUOKA_ERR_INVALID_ARG;
  if (B_e > 0 && (K_sel == nullptr || V_sel == nullptr)) return QUOKA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K_sel) || !aligned16(V_sel) || !aligned16(K_chunk) || !aligned16(V_chunk) ||
      !aligned16(O) || !aligned16(lse))
    return QUOKA_ERR_ALIGNMENT;
  // decode-size chunks need split scratch right after the header
  const size_t dec = use_decode(p, shape) ? attend_decode_ws_bytes(shape->d, shape->H_q, shape->C, B_e) : 0;
  QUOKA_TRY(check_ws(ws, ws_bytes, sizeof(WsHeader) + dec));
  return run_attend(shape, Q, K_sel, V_sel, (int64_t)B_e * shape->d, nullptr, B_e, K_chunk, V_chunk, p, O, lse, ws,
                    sizeof(WsHeader), (cudaStream_t)stream);
}

int quoka_dense_attend(const quoka_shape* shape, const void* Q, const void* K_hist, const void* V_hist,
                       const void* K_chunk, const void* V_chunk, const quoka_params* params, void* O, float* lse,
                       void* ws, size_t ws_bytes, void* stream) {
  QUOKA_TRY(check_shape(shape));
  Params p;
  QUOKA_TRY(read_params(params, shape, &p));
  if (Q == nullptr || K_chunk == nullptr || V_chunk == nullptr || O == nullptr) return QUOKA_ERR_INVALID_ARG;
  if (shape->T > 0 && (K_hist == nullptr || V_hist == nullptr)) return QUOKA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K_hist) || !aligned16(V_hist) || !aligned16(K_chunk) || !aligned16(V_chunk) ||
      !aligned16(O) || !aligned16(lse))
    return QUOKA_ERR_ALIGNMENT;
  const size_t dec = use_decode(p, shape) ? attend_decode_ws_bytes(shape->d, shape->H_q, shape->C, shape->T) : 0;
  QUOKA_TRY(check_ws(ws, ws_bytes, sizeof(WsHeader) + dec));
  return run_attend(shape, Q, K_hist, V_hist, head_stride(shape), nullptr, shape->T, K_chunk, V_chunk, p, O, lse, ws,
                    sizeof(WsHeader), (cudaStream_t)stream);
}

int quoka_chunk_attend(const quoka_shape* shape, const void* Q, const void* K_hist, const void* V_hist,
                       const void* K_chunk, const void* V_chunk, int N_q, int B, const quoka_params* params,
                       void* O, float* lse, int32_t* sel_out, void* ws, size_t ws_bytes, void* stream) {
  QUOKA_TRY(check_shape(shape));
  Params p;
  QUOKA_TRY(read_params(params, shape, &p));
  QUOKA_TRY(check_chunk_args(shape, Q, K_hist, V_hist, K_chunk, V_chunk, N_q, B, O, lse, sel_out));
  const Layout L = make_layout(shape, N_q, B, p);
  QUOKA_TRY(check_ws(ws, ws_bytes, L.total));
  return run_chunk(shape, Q, K_hist, V_hist, K_chunk, V_chunk, N_q, B, p, O, lse, sel_out, ws, L,
                   (cudaStream_t)stream);
}

int quoka_chunk_attend_cached(const quoka_shape* shape, const void* Q, const void* K_hist, const void* V_hist,
                              const void* K_chunk, const void* V_chunk, const float* k_inv_norm,
                              int64_t norm_head_stride, int N_q, int B, const quoka_params* params, void* O,
                              float* lse, int32_t* sel_out, void* ws, size_t ws_bytes, void* stream) {
  QUOKA_TRY(check_shape(shape));
  Params p;
  QUOKA_TRY(read_params(params, shape, &p));
  QUOKA_TRY(check_chunk_args(shape, Q, K_hist, V_hist, K_chunk, V_chunk, N_q, B, O, lse, sel_out));
  QUOKA_TRY(check_norm_cache(shape, k_inv_norm, norm_head_stride, shape->T));
  const Layout L = make_layout(shape, N_q, B, p);
  QUOKA_TRY(check_ws(ws, ws_bytes, L.total));
  KeyCache kc;
  kc.inv = k_inv_norm;
  kc.stride = norm_head_stride;
  return run_chunk(shape, Q, K_hist, V_hist, K_chunk, V_chunk, N_q, B, p, O, lse, sel_out, ws, L,
                   (cudaStream_t)stream, kc);
}

int quoka_workspace_size_varlen(const quoka_varlen_shape* shape, const int64_t* cu_T, const int64_t* cu_C,
                                int N_q, int B, const quoka_params* params, size_t* bytes) {
  if (bytes == nullptr || N_q < 1 || B < 1) return QUOKA_ERR_INVALID_ARG;
  QUOKA_TRY(check_varlen(shape, cu_T, cu_C));
  size_t lane = 0, kept = 0;
  QUOKA_TRY(varlen_lane_bytes(shape, cu_T, cu_C, N_q, B, params, &lane, &kept));
  *bytes = sizeof(WsHeader) + kept + (size_t)varlen_lanes(shape, cu_C) * lane;
  return QUOKA_OK;
}

int quoka_chunk_attend_varlen(const quoka_varlen_shape* shape, const int64_t* cu_T, const int64_t* cu_C,
                              const void* Q, const void* K_hist, const void* V_hist, const void* K_chunk,
                              const void* V_chunk, int N_q, int B, const quoka_params* params, void* O, float* lse,
                              int32_t* sel_out, void* ws, size_t ws_bytes, void* stream) {
  QUOKA_TRY(check_varlen(shape, cu_T, cu_C));
  if (N_q < 1 || B < 1) return QUOKA_ERR_INVALID_ARG;
  const int nseq = shape->nseq;
  const size_t eb = elt_bytes(shape->dtype), d = shape->d;
  size_t lane_bytes = 0, kept_bytes = 0;
  QUOKA_TRY(varlen_lane_bytes(shape, cu_T, cu_C, N_q, B, params, &lane_bytes, &kept_bytes));
  const int lanes = varlen_lanes(shape, cu_C);
  const size_t lane0 = sizeof(WsHeader) + kept_bytes;   // the lanes' slices follow the joint gathered rows
  // Every sequence is checked before the first one is enqueued.
  std::vector<SeqArgs> seqs;
  seqs.reserve(nseq);
  int64_t cu_B = 0;
  for (int s = 0; s < nseq; ++s) {
    SeqArgs a;
    a.shape = seq_shape(shape, cu_T, cu_C, s);
    const int64_t c0 = cu_C[s], t0 = cu_T[s];
    const int64_t B_s = std::min<int64_t>(B, a.shape.T);
    auto off = [](const void* base, size_t elems, size_t bytes) -> const void* {
      return base == nullptr ? nullptr : static_cast<const char*>(base) + elems * bytes;
    };
    a.Q = off(Q, (size_t)shape->H_q * d * c0, eb);
    a.O = const_cast<void*>(off(O, (size_t)shape->H_q * d * c0, eb));
    a.K_chunk = off(K_chunk, (size_t)shape->H_kv * d * c0, eb);
    a.V_chunk = off(V_chunk, (size_t)shape->H_kv * d * c0, eb);
    a.K_hist = a.shape.T > 0 ? off(K_hist, (size_t)shape->H_kv * d * t0, eb) : nullptr;
    a.V_hist = a.shape.T > 0 ? off(V_hist, (size_t)shape->H_kv * d * t0, eb) : nullptr;
    a.lse = lse == nullptr ? nullptr : lse + (size_t)shape->H_q * c0;
    a.sel_out = sel_out == nullptr ? nullptr : sel_out + (size_t)shape->H_kv * cu_B;
    cu_B += B_s;
    if (a.shape.C == 0) continue;
    QUOKA_TRY(read_params(params, &a.shape, &a.p));
    QUOKA_TRY(check_chunk_args(&a.shape, a.Q, a.K_hist, a.V_hist, a.K_chunk, a.V_chunk, N_q, B, a.O, a.lse,
                               a.sel_out));
    a.joint = joint_attention(a.shape, a.p);
    a.kept = 0;
    a.work = seq_work(a.shape, B, !a.joint);
    seqs.push_back(a);
  }
  QUOKA_TRY(check_ws(ws, ws_bytes, lane0 + (size_t)lanes * lane_bytes));
  // the joint sequences' gathered rows, in batch order after the header
  size_t kept_at = sizeof(WsHeader);
  std::vector<AttSeq> joint;
  for (SeqArgs& a : seqs) {
    if (!a.joint) continue;
    const quoka_shape& sh = a.shape;
    AttSeq q{a.Q, a.K_hist, a.V_hist, a.K_chunk, a.V_chunk, head_stride(&sh), sh.T, sh.C, a.O, a.lse};
    if (joint_kept_bytes(sh, B) > 0) {
      a.kept = kept_at;
      q.Kh = at<void>(ws, kept_at);
      q.Vh = at<void>(ws, kept_at + joint_kept_bytes(sh, B) / 2);
      q.h_stride = (int64_t)B * sh.d;
      q.n_hist = B;
      kept_at += joint_kept_bytes(sh, B);
    }
    joint.push_back(q);
  }
  cudaStream_t st = (cudaStream_t)stream;
  if (seqs.empty()) return QUOKA_OK;
  // Longest first onto the least-loaded lane; each lane owns a workspace slice.
  std::vector<int> order(seqs.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = (int)i;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return seqs[a].work > seqs[b].work; });
  std::vector<double> load(lanes, 0.0);
  std::vector<std::vector<int>> plan(lanes);
  for (int i : order) {
    const int l = (int)(std::min_element(load.begin(), load.end()) - load.begin());
    load[l] += seqs[i].work;
    plan[l].push_back(i);
  }
  for (int l = 0; l < lanes; ++l)
    for (int i : plan[l])
      seqs[i].L = make_layout(&seqs[i].shape, N_q, B, seqs[i].p, lane0 + (size_t)l * lane_bytes, !seqs[i].joint);
  // a sequence on its lane: the whole chunk, or (joint) its selection and gather
  auto run_seq = [&](const SeqArgs& a, cudaStream_t lst) -> int {
    KeepOnly keep{a.kept ? at<void>(ws, a.kept) : nullptr,
                  a.kept ? at<void>(ws, a.kept + joint_kept_bytes(a.shape, B) / 2) : nullptr};
    return run_chunk(&a.shape, a.Q, a.K_hist, a.V_hist, a.K_chunk, a.V_chunk, N_q, B, a.p, a.O, a.lse, a.sel_out,
                     ws, a.L, lst, KeyCache(), a.joint ? &keep : nullptr);
  };
  const float scale = seqs[0].p.scale;   // d and the params are the batch's
  auto run_joint = [&]() -> int {
    if (joint.empty()) return QUOKA_OK;
    return cuda_status(launch_attend_tc_varlen(shape->d, joint.data(), (int)joint.size(), shape->H_q, shape->H_kv,
                                               scale, at<WsHeader>(ws, 0), st));
  };
  if (lanes == 1) {
    for (int i : plan[0]) QUOKA_TRY(run_seq(seqs[i], st));
    return run_joint();
  }
  // Fork: lane l > 0 runs on a library stream that first waits for everything
  // enqueued on `stream` so far; lane 0 runs on `stream` itself.  Join: `stream`
  // waits for every lane.  Stream capture follows the fork and the join.
  LaneStreams* ls = nullptr;
  QUOKA_CUDA(lane_streams(&ls));
  std::lock_guard<std::mutex> guard(ls->mu);
  QUOKA_CUDA(cudaEventRecord(ls->fork, st));
  int rc = QUOKA_OK;
  for (int l = 0; l < lanes && rc == QUOKA_OK; ++l) {
    cudaStream_t lst = l == 0 ? st : ls->stream[l - 1];
    if (l > 0 && (rc = cuda_status(cudaStreamWaitEvent(lst, ls->fork, 0))) != QUOKA_OK) break;
    for (int i : plan[l]) {
      rc = run_seq(seqs[i], lst);
      if (rc != QUOKA_OK) break;
    }
  }
  // join every lane that was forked, even after an error, so that a capture stays well formed
  for (int l = 1; l < lanes; ++l) {
    const int j = cuda_status(cudaEventRecord(ls->join[l - 1], ls->stream[l - 1]));
    const int w = j == QUOKA_OK ? cuda_status(cudaStreamWaitEvent(st, ls->join[l - 1], 0)) : j;
    if (rc == QUOKA_OK) rc = w;
  }
  if (rc != QUOKA_OK) return rc;
  return run_joint();   // after the join: every lane's gathered rows are in
}

int quoka_sparse_attend_varlen(const quoka_varlen_shape* shape, const int64_t* cu_B, const int64_t* cu_C,
                               const void* Q, const void* K_sel, const void* V_sel, const void* K_chunk,
                               const void* V_chunk, const quoka_params* params, void* O, float* lse, void* ws,
                               size_t ws_bytes, void* stream) {
  QUOKA_TRY(check_varlen(shape, cu_B, cu_C));
  if (Q == nullptr || K_chunk == nullptr || V_chunk == nullptr || O == nullptr) return QUOKA_ERR_INVALID_ARG;
  const int nseq = shape->nseq;
  if (cu_B[nseq] > 0 && (K_sel == nullptr || V_sel == nullptr)) return QUOKA_ERR_INVALID_ARG;
  const quoka_shape sh0 = seq_shape(shape, cu_B, cu_C, 0);
  Params p;
  QUOKA_TRY(read_params(params, &sh0, &p));
  if (shape->dtype != QUOKA_DTYPE_BF16 || p.engine == QUOKA_ENGINE_SIMT || attend_tc_smem(shape->d) > 227 * 1024)
    return QUOKA_ERR_UNSUPPORTED;
  if (!aligned16(Q) || !aligned16(K_sel) || !aligned16(V_sel) || !aligned16(K_chunk) || !aligned16(V_chunk) ||
      !aligned16(O) || !aligned4(lse))
    return QUOKA_ERR_ALIGNMENT;
  QUOKA_TRY(check_ws(ws, ws_bytes, sizeof(WsHeader)));
  const size_t d = shape->d, eb = 2;
  auto off = [&](const void* base, size_t elems) -> const void* {
    return base == nullptr ? nullptr : static_cast<const char*>(base) + elems * eb;
  };
  std::vector<AttSeq> seqs;
  for (int s = 0; s < nseq; ++s) {
    const int64_t c0 = cu_C[s], b0 = cu_B[s];
    const int C = (int)(cu_C[s + 1] - c0), B_s = (int)(cu_B[s + 1] - b0);
    if (C == 0) continue;
    AttSeq q;
    q.Q = off(Q, (size_t)shape->H_q * d * c0);
    q.O = const_cast<void*>(off(O, (size_t)shape->H_q * d * c0));
    q.Kc = off(K_chunk, (size_t)shape->H_kv * d * c0);
    q.Vc = off(V_chunk, (size_t)shape->H_kv * d * c0);
    q.Kh = B_s > 0 ? off(K_sel, (size_t)shape->H_kv * d * b0) : nullptr;
    q.Vh = B_s > 0 ? off(V_sel, (size_t)shape->H_kv * d * b0) : nullptr;
    q.h_stride = (int64_t)B_s * shape->d;
    q.n_hist = B_s;
    q.C = C;
    q.lse = lse == nullptr ? nullptr : lse + (size_t)shape->H_q * c0;
    seqs.push_back(q);
  }
  if (seqs.empty()) return QUOKA_OK;
  return cuda_status(launch_attend_tc_varlen(shape->d, seqs.data(), (int)seqs.size(), shape->H_q, shape->H_kv,
                                             p.scale, at<WsHeader>(ws, 0), (cudaStream_t)stream));
}

int quoka_append_kv(const quoka_shape* shape, void* K_hist, void* V_hist, const void* K_chunk, const void* V_chunk,
                    void* stream) {
  QUOKA_TRY(check_shape(shape));
  if (!K_hist || !V_hist || !K_chunk || !V_chunk) return QUOKA_ERR_INVALID_ARG;
  if (head_stride(shape) < (int64_t)(shape->T + (int64_t)shape->C) * shape->d) return QUOKA_ERR_INVALID_ARG;
  if (!aligned16(K_hist) || !aligned16(V_hist) || !aligned16(K_chunk) || !aligned16(V_chunk))
    return QUOKA_ERR_ALIGNMENT;
  return cuda_status(launch_append(elt_bytes(shape->dtype), shape->d, K_hist, V_hist, head_stride(shape), shape->T,
                                   K_chunk, V_chunk, shape->H_kv, shape->C, (cudaStream_t)stream));
}

int quoka_append_kv_norms(const quoka_shape* shape, void* K_hist, void* V_hist, const void* K_chunk,
                          const void* V_chunk, float* k_inv_norm, int64_t norm_head_stride, void* stream) {
  QUOKA_TRY(check_norm_cache(shape, k_inv_norm, norm_head_stride, shape->T + shape->C));
  QUOKA_TRY(quoka_append_kv(shape, K_hist, V_hist, K_chunk, V_chunk, stream));
  // the appended keys' norms, from the chunk's own rows (the same values)
  return cuda_status(launch_key_inv_norms(shape->dtype, shape->d, K_chunk, (int64_t)shape->C * shape->d,
                                          shape->H_kv, 0, shape->C, k_inv_norm + shape->T, norm_head_stride,
                                          (cudaStream_t)stream));
}

int quoka_selftest_expire_wait(void* ws, size_t ws_bytes, long long cycles, void* stream) {
  QUOKA_TRY(check_ws(ws, ws_bytes, sizeof(WsHeader)));
  if (cycles < 1) return QUOKA_ERR_INVALID_ARG;
  return cuda_status(launch_expire_wait(at<WsHeader>(ws, 0), cycles, (cudaStream_t)stream));
}

int quoka_get_last_device_error(void* ws, void* stream) {
  if (ws == nullptr) return QUOKA_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  WsHeader h;
  if (cudaMemcpyAsync(&h, ws, 8, cudaMemcpyDeviceToHost, st) != cudaSuccess) return QUOKA_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, 8, st) != cudaSuccess) return QUOKA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return QUOKA_ERR_CUDA;
  return (int)h.err;
}

}  // extern "C"
