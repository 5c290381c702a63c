/*
 * quoka.h -- C ABI of libquoka.so: QUOKA per-chunk KV selection plus sparse
 * attention for chunked prefill, on GB300 (sm_103a).
 *
 * Method sources (page title, section):
 *   [P1] "QUOKA: Query-Oriented KV Selection For Efficient LLM Prefill"
 *        (paper summary): "Transformers and Attention", "Chunked prefill",
 *        "Attention Sparsity and Sparse Attention", "QUOKA Method",
 *        "Query Subselection", "Scoring via Cosine Similarity",
 *        "Aggregation Across Queries and KV Groups", "Chunked Prefill with QUOKA".
 *   [P2] "QUOKA Explained: Choosing Which KV History Attention Should Read":
 *        "Pick the queries that disagree with the crowd", "Letting those
 *        queries score the history", "Why take the maximum", "From scores to
 *        a smaller KV set", "A wrinkle: grouped-query attention", "MEAN and
 *        MAX do different jobs".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Tensors are row-major and contiguous unless a stride says otherwise:
 *   Q        [H_q,  C, d]   chunk queries
 *   K_hist   [H_kv, T, d]   cached history keys; consecutive KV heads are
 *   V_hist   [H_kv, T, d]   kv_head_stride elements apart (>= T*d, so a
 *                           preallocated cache can grow in place)
 *   K_chunk  [H_kv, C, d]   the chunk's own keys / values
 *   V_chunk  [H_kv, C, d]
 *   O        [H_q,  C, d]   output, same element type as Q
 * Query head h reads KV head h / (H_q / H_kv).  The element type of every
 * tensor argument is shape->dtype (bf16 or fp32); scores and lse are fp32;
 * index arrays are int32.
 *
 * Pointers: every tensor pointer is a DEVICE pointer (or managed memory)
 * owned by the caller and 16-byte aligned (the lse and sel_out outputs of
 * quoka_chunk_attend and its ragged form: 4-byte); the library never allocates,
 * frees or synchronises on these paths.  `stream` is a cudaStream_t (NULL is
 * the legacy default stream); every call only enqueues work on it and
 * returns.  Results are valid once the stream reaches that point.
 *
 * Workspace: calls that take (ws, ws_bytes) use caller-owned device scratch of
 * at least quoka_workspace_size() bytes, 256-byte aligned.  Its first word is
 * the sticky device error status (see quoka_get_last_device_error); zero it
 * once (cudaMemset) before first use.  Calls sharing one workspace must be
 * ordered on one stream.
 *
 * Errors: every function returns a quoka_status.  Argument checks happen on
 * the host before anything is enqueued; a non-OK return means nothing was
 * enqueued, except QUOKA_ERR_CUDA (a launch failed).  Errors found by the GPU
 * (an expired bounded wait) are recorded in the workspace error word.
 */
#ifndef QUOKA_H_
#define QUOKA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QUOKA_OK = 0,
  QUOKA_ERR_INVALID_ARG = 1,   /* a size, pointer or mode is out of range */
  QUOKA_ERR_UNSUPPORTED = 2,   /* valid, but outside what the kernels handle (e.g. d not 64/128) */
  QUOKA_ERR_WORKSPACE = 3,     /* ws is NULL, misaligned or smaller than required */
  QUOKA_ERR_ALIGNMENT = 4,     /* a tensor pointer is not 16-byte aligned */
  QUOKA_ERR_CUDA = 5,          /* a CUDA runtime call or kernel launch failed */
  QUOKA_ERR_TIMEOUT = 6,       /* device side: a bounded wait expired (kernel exited early) */
  QUOKA_ERR_DEVICE = 7         /* device side: a kept position outside [0, T) was skipped */
} quoka_status;

typedef enum { QUOKA_DTYPE_BF16 = 0, QUOKA_DTYPE_FP32 = 1 } quoka_dtype;

/* How scores of the query heads of one KV group are pooled
 * ([P1] "Aggregation Across Queries and KV Groups"; [P2] "A wrinkle:
 * grouped-query attention", "MEAN and MAX do different jobs").
 *  MEAN_PREAGG: one selected token set per KV group (the group's per-head
 *    cosines to their mean queries are averaged before the N_q least
 *    similar tokens are kept); the normalised query heads of each kept token
 *    are averaged (not re-normalised) and that one row scores the keys, so
 *    a key's score is the maximum over tokens of the head-averaged cosine.
 *  MAX: one selected token set per query head; every selected row of every
 *    head of the group scores the keys and the maximum is taken over all
 *    of them. */
typedef enum { QUOKA_GQA_MEAN_PREAGG = 0, QUOKA_GQA_MAX = 1 } quoka_gqa_pool;

/* Which kernel family runs the scoring and attention stages.  AUTO picks the
 * tensor-core (tcgen05) kernels for bf16 where they exist and the CUDA-core
 * kernels otherwise; SIMT forces the CUDA-core kernels (fp32 always uses them). */
typedef enum { QUOKA_ENGINE_AUTO = 0, QUOKA_ENGINE_SIMT = 1, QUOKA_ENGINE_TENSOR = 2 } quoka_engine;

typedef struct {
  int64_t kv_head_stride;  /* elements between KV heads of K_hist / V_hist; 0 means T*d */
  int32_t H_q;             /* query heads, >= 1, multiple of H_kv */
  int32_t H_kv;            /* KV heads, >= 1 */
  int32_t C;               /* chunk length (queries), 1 .. 8192 */
  int32_t T;               /* history length (cached keys), >= 0 */
  int32_t d;               /* head dim, 64 or 128 */
  int32_t dtype;           /* quoka_dtype */
} quoka_shape;

/* Variants of the key score, OR-ed into quoka_params.flags.  The pages report
 * both as ablations of the method ([P1] "Scoring via Cosine Similarity":
 * cosine against the plain dot product; [P1] "Aggregation Across Queries and
 * KV Groups", [P2] "Why take the maximum": the maximum against the mean over
 * the selected queries).  0 is the method as published.  They change the key
 * score only: query subselection is always on the cosine to the mean query,
 * and attention is unchanged.
 *  SCORE_DOT:  score rows and keys are not normalised: r . k_t.  With
 *              MEAN_PREAGG the pre-aggregated row is the mean of the raw
 *              query heads.
 *  QUERY_MEAN: the selected tokens are aggregated by their mean instead of
 *              the maximum.  With QUOKA_GQA_MAX each head's tokens are
 *              averaged and the maximum over the group's heads is kept. */
enum { QUOKA_FLAG_SCORE_DOT = 1, QUOKA_FLAG_QUERY_MEAN = 2 };

typedef struct {
  int32_t gqa_pool;        /* quoka_gqa_pool */
  int32_t engine;          /* quoka_engine */
  float softmax_scale;     /* <= 0 means 1/sqrt(d) */
  int32_t flags;           /* 0, or an OR of QUOKA_FLAG_*; other bits must be 0 */
} quoka_params;

/* Human-readable name of a status code (static storage). */
const char* quoka_status_string(int status);

/* Bytes of workspace that quoka_chunk_attend needs for this problem; the
 * same size also covers every single-stage call on the same shape.
 * N_q and B as for quoka_chunk_attend.  Writes *bytes; host only. */
int quoka_workspace_size(const quoka_shape* shape, int N_q, int B, const quoka_params* params,
                         size_t* bytes);

/* Query subselection ([P1] "Query Subselection"; [P2] "Pick the queries that
 * disagree with the crowd").  Per query head the mean query M_q of the
 * chunk's C raw queries is formed and every query's cosine to it computed
 * (norms clamped at 1e-12); the N_q' = min(N_q, C) queries with the smallest
 * cosine (largest -CosSim) are kept, ties to the lower position.
 * q_idx: int32 [H_sel, N_q'] written in ascending order, where H_sel = H_q
 * for QUOKA_GQA_MAX (per head) and H_kv for QUOKA_GQA_MEAN_PREAGG (per group,
 * on the cosine averaged over the group's heads).  Uses ws. */
int quoka_select_queries(const quoka_shape* shape, const void* Q, int N_q, const quoka_params* params,
                         int32_t* q_idx, void* ws, size_t ws_bytes, void* stream);

/* quoka_select_queries without a workspace (the paper has no counterpart: this
 * is a calling convention, not a step of the method).  For callers that
 * cannot provide device scratch memory at all -- inference-engine plugins
 * whose enqueue path may not allocate, and runtimes that plan every byte of
 * device memory ahead of time -- the scratch lives in a 4 MiB device array
 * owned by the library, which every GPU that loads libquoka.so holds until
 * the process exits.  Same arguments, checks, layout and results as
 * quoka_select_queries, minus (ws, ws_bytes); nothing is allocated.
 * Limit: max pooling uses only the array's 256-byte error header.  Mean
 * pooling keeps its per-head cosines in the array (a clustered pass per query
 * head, then a clustered select per KV group) when 256 + 4*H_q*C bytes (the
 * cosines rounded up to 256) fit in 4 MiB; otherwise it runs one clustered
 * launch over whole groups, whose shared memory must stay within 160 KB
 * (about (2 + G)*C/2 + 2*G*d*4 bytes plus 64 KB of staging, G = H_q / H_kv),
 * else the call returns QUOKA_ERR_UNSUPPORTED.  The first call on a device
 * looks up the array's device address (make that first call before any
 * stream capture).  Every call shares the one array, which keeps the last
 * call's contents: calls that overlap on the GPU (different streams or host
 * threads) race and must be serialised by the caller.  A device-side failure
 * (an expired bounded wait) is recorded in the array's header, which the C
 * ABI does not expose: callers that need device errors reported use
 * quoka_select_queries with a workspace and quoka_get_last_device_error. */
int quoka_select_queries_noalloc(const quoka_shape* shape, const void* Q, int N_q, const quoka_params* params,
                                 int32_t* q_idx, void* stream);

/* Cosine scoring plus aggregation ([P1] "Scoring via Cosine Similarity",
 * "Aggregation Across Queries and KV Groups"; [P2] "Letting those queries
 * score the history", "Why take the maximum").  For every KV group g and
 * history key t < T:
 *   scores[g, t] = max over the group's scoring rows r of  r . k_t / |k_t|
 * where the rows are the normalised selected queries of every head of g
 * (MAX) or their head average per selected token (MEAN_PREAGG).  Products
 * are accumulated in fp32.  params->flags selects the ablation variants
 * (QUOKA_FLAG_*).  q_idx as written by quoka_select_queries with the
 * same N_q and pooling.  scores: fp32 [H_kv, T].  Uses ws. */
int quoka_score_keys(const quoka_shape* shape, const void* Q, const int32_t* q_idx, int N_q,
                     const void* K_hist, const quoka_params* params, float* scores,
                     void* ws, size_t ws_bytes, void* stream);

/* Key-norm cache ([P1] "Chunked Prefill with QUOKA": the keys enter the cache
 * once and are scored by every later chunk, so their norms can be stored when
 * they are written).  k_inv_norm[g * norm_head_stride + t] =
 * 1 / max(|K_hist[g, t]|, 1e-12) in fp32 for t in [t0, t1), t1 <= T.
 * k_inv_norm: device fp32, 4-byte aligned, norm_head_stride >= t1. */
int quoka_key_inv_norms(const quoka_shape* shape, const void* K_hist, int t0, int t1, float* k_inv_norm,
                        int64_t norm_head_stride, void* stream);

/* quoka_score_keys with the key norms taken from the cache (norm_head_stride
 * >= T) instead of recomputed from the keys; the cache must hold the norms of
 * exactly these keys (quoka_key_inv_norms / quoka_append_kv_norms).  Scores
 * agree with quoka_score_keys to fp32 rounding of the norms. */
int quoka_score_keys_cached(const quoka_shape* shape, const void* Q, const int32_t* q_idx, int N_q,
                            const void* K_hist, const float* k_inv_norm, int64_t norm_head_stride,
                            const quoka_params* params, float* scores, void* ws, size_t ws_bytes, void* stream);

/* Top-B history keys per KV head ([P2] "From scores to a smaller KV set").
 * Reads scores fp32 [H_kv, T] (shape->H_kv, shape->T); writes sel int32
 * [H_kv, B_e], B_e = min(B, T), the positions of the B_e largest scores in
 * ascending position order, ties to the lower position (-0.0 equals 0.0).
 * Scores must not be NaN.  Uses ws. */
int quoka_topk(const quoka_shape* shape, const float* scores, int B, int32_t* sel,
               void* ws, size_t ws_bytes, void* stream);

/* Gather the selected rows: K_sel[g, j] = K_hist[g, sel[g, j]], same for V
 * ([P2] "From scores to a smaller KV set": the value comes with its key).
 * sel int32 [H_kv, B_e], every entry in [0, T); K_sel, V_sel [H_kv, B_e, d]
 * contiguous, dtype of the shape.  An entry outside [0, T) is checked on the
 * device and never dereferenced: its rows are written as zeros.  (This call
 * has no workspace, so it cannot record the error; inside quoka_chunk_attend
 * the same check records QUOKA_ERR_DEVICE in the workspace header.) */
int quoka_gather(const quoka_shape* shape, const void* K_hist, const void* V_hist, const int32_t* sel,
                 int B_e, void* K_sel, void* V_sel, void* stream);

/* Attention over the reduced set ([P1] "Transformers and Attention",
 * "Chunked prefill", "QUOKA Method"; [P2] "MEAN and MAX do different jobs":
 * the original query heads attend).  For query head h, chunk row c:
 *   O[h, c] = softmax_j(scale * Q[h, c] . k_j) v_j over the keys
 *   k = [K_sel[g, 0..B_e) ; K_chunk[g, 0..c]]   (causal within the chunk)
 * K_sel, V_sel [H_kv, B_e, d] contiguous (B_e may be 0).  lse, if not NULL,
 * receives fp32 [H_q, C] natural-log softmax denominators of the scaled
 * logits.  Uses ws: the error word and, for chunks of at most 32 / G queries
 * (decode), scratch for the split-key partial results (quoka_workspace_size
 * covers it). */
int quoka_sparse_attend(const quoka_shape* shape, const void* Q, const void* K_sel, const void* V_sel,
                        int B_e, const void* K_chunk, const void* V_chunk, const quoka_params* params,
                        void* O, float* lse, void* ws, size_t ws_bytes, void* stream);

/* One chunk of QUOKA chunked prefill end to end ([P1] "QUOKA Method",
 * "Chunked Prefill with QUOKA"): select queries, score the history, keep the
 * top-B keys per KV head, attend to them plus the causal chunk.  T = 0 or
 * B >= T skips selection and attends to the whole history.  sel_out, if not
 * NULL, receives int32 [H_kv, min(B, T)] (ascending); lse as above. */
int quoka_chunk_attend(const quoka_shape* shape, const void* Q, const void* K_hist, const void* V_hist,
                       const void* K_chunk, const void* V_chunk, int N_q, int B,
                       const quoka_params* params, void* O, float* lse, int32_t* sel_out,
                       void* ws, size_t ws_bytes, void* stream);

/* Shape of a ragged batch: nseq sequences, each with its own chunk length
 * C_s and history length T_s, sharing the head layout and element type. */
typedef struct {
  int32_t nseq;            /* sequences, >= 1 */
  int32_t H_q;             /* as quoka_shape */
  int32_t H_kv;
  int32_t d;
  int32_t dtype;
  int32_t reserved;        /* must be 0 */
} quoka_varlen_shape;

/* Workspace bytes for quoka_chunk_attend_varlen: the 256-byte error header,
 * then the kept K and V rows of every sequence that attends in the joint
 * launch and selects keys (0 < B < T_s; 2 * H_kv * B * d elements each,
 * every block rounded up to 256 bytes), then one slice per stream lane (one
 * lane per sequence with C_s > 0, at most 8), each slice the largest
 * single-sequence requirement of the batch without those rows.
 * cu_T, cu_C as for quoka_chunk_attend_varlen. */
int quoka_workspace_size_varlen(const quoka_varlen_shape* shape, const int64_t* cu_T, const int64_t* cu_C,
                                int N_q, int B, const quoka_params* params, size_t* bytes);

/* quoka_chunk_attend over a ragged batch in one call ([P1] "Chunked Prefill
 * with QUOKA": every sequence's chunk is processed against its own cache; the
 * sequences share nothing).  cu_T and cu_C are HOST int64 arrays of nseq + 1
 * prefix sums (cu[0] = 0, non-decreasing): sequence s has
 * T_s = cu_T[s+1] - cu_T[s] history keys and C_s = cu_C[s+1] - cu_C[s] chunk
 * queries (C_s = 0: the sequence is skipped; each C_s <= 8192).
 * Packed tensors, sequence-major: every sequence's block is laid out exactly
 * as quoka_chunk_attend's tensors and the blocks are concatenated, so
 * sequence s's
 *   Q, O        start at element H_q  * d * cu_C[s]   ([H_q,  C_s, d])
 *   K/V_chunk   start at element H_kv * d * cu_C[s]   ([H_kv, C_s, d])
 *   K/V_hist    start at element H_kv * d * cu_T[s]   ([H_kv, T_s, d], heads T_s * d apart)
 *   lse         starts at H_q * cu_C[s]               (fp32 [H_q, C_s]; may be NULL)
 *   sel_out     starts at H_kv * cu_B[s], with cu_B the prefix sums of
 *               B_s = min(B, T_s)                      (int32 [H_kv, B_s]; may be NULL;
 *               a skipped sequence keeps its rows, left unwritten).
 * lse and sel_out need only 4-byte alignment; the other tensors 16 bytes.
 * N_q, B and params apply to every sequence.  Every sequence is checked before
 * anything is enqueued.  The sequences then go through the same kernels as
 * quoka_chunk_attend on up to 8 stream lanes: `stream` itself and
 * library-owned streams (created once per device) that first wait for
 * everything enqueued on `stream` so far; `stream` then waits for every lane,
 * so the call behaves as one unit of work on `stream` (and stream capture
 * records the fork and the join).  Each lane uses its own slice of ws; the
 * error header is shared.  Sequences whose attention runs on the tensor cores
 * (bf16, G * C_s > 32 or the tensor engine forced) stop on their lane after
 * the gather: after the join, one persistent attention launch per 16 such
 * sequences, on `stream`, attends for all of them (as
 * quoka_sparse_attend_varlen does).  The results are those of
 * quoka_chunk_attend on each sequence, bit for bit.  Concurrent calls from
 * several host threads are serialised on the lane streams. */
int quoka_chunk_attend_varlen(const quoka_varlen_shape* shape, const int64_t* cu_T, const int64_t* cu_C,
                              const void* Q, const void* K_hist, const void* V_hist, const void* K_chunk,
                              const void* V_chunk, int N_q, int B, const quoka_params* params, void* O, float* lse,
                              int32_t* sel_out, void* ws, size_t ws_bytes, void* stream);

/* quoka_sparse_attend over a ragged batch ([P1] "Chunked Prefill with QUOKA":
 * each sequence attends to its own kept rows and its causal chunk): one
 * persistent tensor-core launch per 16 sequences deals the work items (query
 * tile x head pair) of every sequence to one CTA per SM, sequence by
 * sequence (the sequences with the longest items first, each sequence's
 * longest items first), so that a sequence's K/V rows stay in L2 while its
 * items run.  cu_B and cu_C are HOST int64 arrays of nseq + 1 prefix sums
 * (cu[0] = 0, non-decreasing): sequence s has
 * B_s = cu_B[s+1] - cu_B[s] kept rows (0 allowed) and C_s = cu_C[s+1] - cu_C[s]
 * queries (0: the sequence is skipped; each C_s <= 8192).  Packed tensors,
 * sequence-major:
 *   Q, O          start at element H_q  * d * cu_C[s]   ([H_q,  C_s, d])
 *   K_sel, V_sel  start at element H_kv * d * cu_B[s]   ([H_kv, B_s, d])
 *   K/V_chunk     start at element H_kv * d * cu_C[s]   ([H_kv, C_s, d])
 *   lse           starts at H_q * cu_C[s]               (fp32 [H_q, C_s]; may be NULL)
 * lse needs 4-byte alignment, the other tensors 16 bytes.  bf16 only, and
 * not with QUOKA_ENGINE_SIMT (QUOKA_ERR_UNSUPPORTED); of params only
 * softmax_scale is read.  ws: the 256-byte error header.  Each sequence's
 * O and lse are those of quoka_sparse_attend with QUOKA_ENGINE_TENSOR on that
 * sequence, bit for bit. */
int quoka_sparse_attend_varlen(const quoka_varlen_shape* shape, const int64_t* cu_B, const int64_t* cu_C,
                               const void* Q, const void* K_sel, const void* V_sel, const void* K_chunk,
                               const void* V_chunk, const quoka_params* params, void* O, float* lse, void* ws,
                               size_t ws_bytes, void* stream);

/* quoka_chunk_attend with the history's key norms from the cache (as
 * quoka_score_keys_cached). */
int quoka_chunk_attend_cached(const quoka_shape* shape, const void* Q, const void* K_hist, const void* V_hist,
                              const void* K_chunk, const void* V_chunk, const float* k_inv_norm,
                              int64_t norm_head_stride, int N_q, int B, const quoka_params* params, void* O,
                              float* lse, int32_t* sel_out, void* ws, size_t ws_bytes, void* stream);

/* Dense chunked-prefill attention over every history key plus the causal
 * chunk ([P1] "Chunked prefill"): the reference QUOKA is measured against.
 * Arguments as quoka_chunk_attend without the selection; ws as for
 * quoka_sparse_attend. */
int quoka_dense_attend(const quoka_shape* shape, const void* Q, const void* K_hist, const void* V_hist,
                       const void* K_chunk, const void* V_chunk, const quoka_params* params,
                       void* O, float* lse, void* ws, size_t ws_bytes, void* stream);

/* Append the chunk's keys and values to the cache ([P2] "MEAN and MAX do
 * different jobs": nothing is evicted): K_hist[g, T + c] = K_chunk[g, c] and
 * likewise V, for c < C.  Requires kv_head_stride >= (T + C) * d. */
int quoka_append_kv(const quoka_shape* shape, void* K_hist, void* V_hist, const void* K_chunk,
                    const void* V_chunk, void* stream);

/* quoka_append_kv, and the appended keys' entries of the key-norm cache:
 * k_inv_norm[g * norm_head_stride + T + c] = 1 / max(|K_chunk[g, c]|, 1e-12)
 * for c < C (norm_head_stride >= T + C). */
int quoka_append_kv_norms(const quoka_shape* shape, void* K_hist, void* V_hist, const void* K_chunk,
                          const void* V_chunk, float* k_inv_norm, int64_t norm_head_stride, void* stream);

/* Which kernel family a stage runs for this shape and params:
 * QUOKA_ENGINE_TENSOR (tcgen05 tensor cores) or QUOKA_ENGINE_SIMT (CUDA
 * cores).  stage: 0 = key scoring, 1 = attention.  Returns a negative
 * quoka_status if the shape, params or stage are invalid.  Host only. */
int quoka_stage_engine(const quoka_shape* shape, const quoka_params* params, int stage);

/* Description of the CUDA error behind the calling thread's most recent
 * QUOKA_ERR_CUDA ("no error" if there was none).  Static storage. */
const char* quoka_last_cuda_error_string(void);

/* Number of CUDA kernels this library has enqueued in this process so far
 * (diagnostics: lets a caller count the launches of a timed region). */
uint64_t quoka_launch_count(void);

/* Self-test of device-side failure detection: enqueues a kernel whose one
 * wait can never be satisfied; the wait gives up after `cycles` SM clock
 * cycles, records QUOKA_ERR_TIMEOUT in the workspace error word and the
 * kernel returns normally (no fault, no hang; the context stays usable).
 * Read the result with quoka_get_last_device_error. */
int quoka_selftest_expire_wait(void* ws, size_t ws_bytes, long long cycles, void* stream);

/* Synchronises `stream`, returns the device error recorded in ws (QUOKA_OK
 * if none) and clears it.  Returns QUOKA_ERR_CUDA if the synchronisation or
 * the read fails. */
int quoka_get_last_device_error(void* ws, void* stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* QUOKA_H_ */
