// Internal launchers (host side) of the QUOKA kernels.  dtype: 0 = bf16,
// 1 = fp32 (quoka_dtype); d: 64 or 128.  Every launcher only enqueues on `st`
// and returns the launch status.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

namespace quoka {

// Kernels enqueued by this library in this process (read by quoka_launch_count).
extern std::atomic<unsigned long long> g_launch_count;
inline void count_launches(unsigned n) { g_launch_count.fetch_add(n, std::memory_order_relaxed); }

cudaError_t launch_select_queries(int dtype, int d, const void* Q, int H_q, int G_avg, int C, int n_sel,
                                  int32_t* q_idx, float* qnorm, float* qpart, float* qcos, cudaStream_t st);

cudaError_t launch_build_operand(int dtype, int d, const void* Q, const int32_t* q_idx, int H_kv, int C, int G,
                                 int n, int mode, float* op_f32, __nv_bfloat16* op_bf, float* op_scale,
                                 cudaStream_t st);

cudaError_t launch_score_simt(int dtype, int d, const void* K, int64_t head_stride, int H_kv, int T_len,
                              const float* op_f32, int R, float* scores, cudaStream_t st);

cudaError_t launch_topk(const float* scores, int H_kv, int T_len, int B_e, int32_t* sel, cudaStream_t st);

cudaError_t launch_gather(int elt_bytes, int d, const void* K, const void* V, int64_t head_stride, const int32_t* sel,
                          int H_kv, int B_e, void* Ks, void* Vs, cudaStream_t st);

cudaError_t launch_append(int elt_bytes, int d, void* K, void* V, int64_t head_stride, int T_len, const void* Kc,
                          const void* Vc, int H_kv, int C, cudaStream_t st);

cudaError_t launch_attend_simt(int dtype, int d, const void* Q, const void* Kh, const void* Vh, int64_t h_stride,
                               int n_hist, const void* Kc, const void* Vc, int H_q, int C, int G, float scale,
                               void* O, float* lse, cudaStream_t st);

}  // namespace quoka
