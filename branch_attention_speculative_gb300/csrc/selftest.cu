// Self-test of the device-side failure path: one CTA waits, with the same
// bounded mbarrier wait every tcgen05 kernel uses, on a barrier that nothing
// will ever complete.  The wait gives up after `cycles` SM clocks, records
// BA_DEV_TIMEOUT in the status word and the kernel returns normally, so the
// context stays usable.  No trap, no fault, no endless loop.
#include "kernels.h"
#include "tc.cuh"

namespace {

__global__ void wait_timeout_kernel(unsigned int* status, long long cycles) {
  __shared__ __align__(8) unsigned long long bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);  // expects one arrival that never comes
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, status, &abort_flag, cycles);
  __syncthreads();
}

}  // namespace

cudaError_t ba_launch_selftest_wait_timeout(unsigned int* status, long long cycles, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(status, cycles);
  return cudaGetLastError();
}
