// Failure-detection self-test (sm_103a).
//
// Every wait in the library's kernels is bounded: on expiry it records a code
// in the device error flag and the kernel leaves cleanly, so the context stays
// usable and convrot_check_device_error() reports CONVROT_ERR_TIMEOUT.  This
// kernel exercises exactly that path without faulting or hanging anything: it
// waits on an mbarrier that nothing will ever arrive on, with a short budget.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace convrot {

__global__ void selftest_wait_kernel(int* err, long long budget) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  // No thread arrives on `bar` and no copy targets it: the wait runs out.
  if (threadIdx.x == 0) mbar_wait_budget(&bar, 0, err, DEVERR_SELFTEST, budget);
}

cudaError_t launch_selftest_wait(int* err, long long budget, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(err, budget);
  return cudaGetLastError();
}

}  // namespace convrot
