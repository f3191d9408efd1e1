// Debug kernel that exercises the bounded-wait path: it waits on an mbarrier nothing will ever
// arrive on, gives up after `limit_ns`, records the timeout in the status word and returns.
#include <cuda_runtime.h>

#include "launch.h"

namespace afx {

__global__ void wait_timeout_kernel(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(&bar), 0)) {
      if (globaltimer_ns() - t0 > limit_ns) {
        atomicOr(status, kDevTimeout);
        break;
      }
    }
  }
  __syncthreads();
}

cudaError_t launch_wait_timeout(uint64_t limit_ns, int* status, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace afx
