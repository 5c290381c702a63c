// The library-owned device scratch of quoka_select_queries_noalloc (the entry
// point itself is in quoka_api.cu, next to quoka_select_queries, whose checks,
// error reporting and launch sequence it shares).
//
// Some callers cannot hand the library any device memory beyond the inputs
// and outputs: inference-engine plugins whose enqueue path may not allocate,
// and runtimes that plan every byte of device memory ahead of time and have
// no spare buffer to pass.  For them the query-selection kernels' scratch
// (an error header, row norms, partial column sums, cosines) lives in this
// file-scope __device__ array, which every GPU that loads the library holds
// until the process exits.
//
// In host code the array's name is a host-side stand-in, not a device
// address, so its address is looked up once per device, with that device
// current, by the first call made on the device (make that first call before
// any stream capture).  All calls share the one array and it keeps the last
// call's contents; calls that overlap on the GPU race on it.
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace quoka {
namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

cudaError_t noalloc_scratch(void** base) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *base = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace quoka
