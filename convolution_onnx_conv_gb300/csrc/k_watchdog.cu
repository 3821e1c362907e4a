// Self-test of the bounded mbarrier wait that every kernel uses: one thread waits on a
// barrier that nobody arrives at; the wait must give up after `budget` cycles and set the
// timeout bit in *status, leaving the context usable.
#include "convf_internal.h"
#include "ptx.cuh"

namespace convf {

__global__ void watchdog_selftest_kernel(int32_t* status, long long budget) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, status, budget);
}

cudaError_t launch_watchdog_selftest(int32_t* status, long long budget, cudaStream_t stream) {
  watchdog_selftest_kernel<<<1, 32, 0, stream>>>(status, budget);
  return cudaGetLastError();
}

}  // namespace convf
