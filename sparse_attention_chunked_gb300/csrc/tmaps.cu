// Host-side TMA tensor-map encoding through the driver entry point (no libcuda link).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "launch.h"

namespace quoka {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 tensor of extents {d0 (innermost, contiguous), d1, d2}; strides in bytes
// for dims 1 and 2 (multiples of 16); box {box0, box1, 1}; 128-byte swizzle
// (box0 * 2 must be <= 128).  Out-of-range elements read as zero.
cudaError_t make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                              uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1) {
  auto fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1, stride2};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Raises a kernel's dynamic shared-memory limit on the current device, once
// per (kernel, device) unless a larger size is asked for later.
cudaError_t ensure_smem(const void* func, size_t bytes) {
  // The 48 KB default covers static plus dynamic shared memory, so a kernel
  // with static shared memory needs the opt-in below 48 KB of dynamic too.
  if (bytes == 0) return cudaSuccess;
  struct Entry {
    const void* func;
    int dev;
    size_t bytes;
  };
  static Entry table[64];
  static int used = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (table[i].func == func && table[i].dev == dev && table[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < used; ++i)
    if (table[i].func == func && table[i].dev == dev) {
      table[i].bytes = bytes;
      return cudaSuccess;
    }
  if (used < 64) table[used++] = Entry{func, dev, bytes};
  return cudaSuccess;
}

}  // namespace quoka
