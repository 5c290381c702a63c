// Self-test of the bounded wait used by every tcgen05 / TMA kernel: one CTA
// waits on an mbarrier that nothing will ever arrive on.  The wait must give
// up after `limit` cycles, record QUOKA_ERR_TIMEOUT in the workspace header and
// let the kernel return, leaving the CUDA context usable.
#include "launch.h"
#include "tc_common.cuh"

namespace quoka {

__global__ void k_expire_wait(WsHeader* hdr, long long limit) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    abort = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) tc::mbar_wait(&bar, 0, &abort, hdr, 0x7e57, limit);   // never completes: must time out
  __syncthreads();
}

cudaError_t launch_expire_wait(WsHeader* hdr, long long limit, cudaStream_t st) {
  k_expire_wait<<<1, 32, 0, st>>>(hdr, limit);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace quoka
