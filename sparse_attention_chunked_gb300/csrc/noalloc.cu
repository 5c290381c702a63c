// quoka_select_queries_noalloc: query subselection with its scratch in a
// fixed, library-owned device buffer instead of a caller-provided workspace.
//
// Some callers cannot hand the library any device memory beyond the inputs
// and outputs: inference-engine plugins whose enqueue path may not allocate,
// and runtimes that plan every byte of device memory ahead of time and have
// no spare buffer to pass.  For them this entry point keeps the scratch of the
// query-selection kernels (row norms, partial column sums, cosines) in a
// file-scope __device__ array of kNoAllocScratchBytes, which every GPU that
// loads the library holds until the process exits.
//
// The device address of that array is looked up once per device, with the
// device current, by the first call made on that device; make that first call
// before any stream capture.  All calls share the one array and it keeps the
// contents of the last call (the kernels write every element they later read,
// so nothing needs clearing); calls that overlap on the GPU (different
// streams, or several host threads) race on it and must be serialised by the
// caller.
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "quoka.h"

namespace quoka {
namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;   // 4 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QUOKA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return QUOKA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return QUOKA_OK;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace quoka

extern "C" int quoka_select_queries_noalloc(const quoka_shape* s, const void* Q, int N_q, const quoka_params* params,
                                            int32_t* q_idx, void* stream) {
  using namespace quoka;
  if (s == nullptr || Q == nullptr || q_idx == nullptr || N_q < 1) return QUOKA_ERR_INVALID_ARG;
  if (s->H_q < 1 || s->H_kv < 1 || s->H_q % s->H_kv != 0 || s->C < 1) return QUOKA_ERR_INVALID_ARG;
  if (s->dtype != QUOKA_DTYPE_BF16 && s->dtype != QUOKA_DTYPE_FP32) return QUOKA_ERR_INVALID_ARG;
  if (s->d != 64 && s->d != 128) return QUOKA_ERR_UNSUPPORTED;
  if (s->C > 8192) return QUOKA_ERR_UNSUPPORTED;
  int gqa = QUOKA_GQA_MEAN_PREAGG;
  if (params != nullptr) {
    if (params->gqa_pool != QUOKA_GQA_MEAN_PREAGG && params->gqa_pool != QUOKA_GQA_MAX) return QUOKA_ERR_INVALID_ARG;
    if ((params->flags & ~(QUOKA_FLAG_SCORE_DOT | QUOKA_FLAG_QUERY_MEAN)) != 0) return QUOKA_ERR_INVALID_ARG;
    gqa = params->gqa_pool;
  }
  if (((uintptr_t)Q & 15u) != 0 || ((uintptr_t)q_idx & 15u) != 0) return QUOKA_ERR_ALIGNMENT;
  // scratch layout, as in the workspace: row norms | partial column sums | cosines
  const size_t H_q = s->H_q, C = s->C, d = s->d, nblk = (C + 63) / 64;
  const size_t off_norm = 0;
  const size_t off_part = align256(off_norm + H_q * C * 4);
  const size_t off_cos = align256(off_part + H_q * nblk * d * 4);
  const size_t need = align256(off_cos + H_q * C * 4);
  if (need > kNoAllocScratchBytes) return QUOKA_ERR_UNSUPPORTED;   // beyond the static scratch
  void* base = nullptr;
  const int rc = scratch_address(&base);
  if (rc != QUOKA_OK) return rc;
  char* b = static_cast<char*>(base);
  const int n = N_q < s->C ? N_q : s->C;
  const int G_avg = gqa == QUOKA_GQA_MAX ? 1 : s->H_q / s->H_kv;
  const cudaError_t e = launch_select_queries(s->dtype, s->d, Q, s->H_q, G_avg, s->C, n, q_idx,
                                              reinterpret_cast<float*>(b + off_norm), reinterpret_cast<float*>(b + off_part),
                                              reinterpret_cast<float*>(b + off_cos), nullptr, (cudaStream_t)stream);
  return e == cudaSuccess ? QUOKA_OK : QUOKA_ERR_CUDA;
}
