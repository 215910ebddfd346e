// Self-test of the bounded device-side wait that every tensor-core kernel of
// this library uses (mbar_wait in tc.cuh, the device flag of common.cuh).
//
// One CTA initialises an mbarrier that nothing ever arrives on and waits for
// it with the kernels' bounded wait and a caller-given poll budget. The wait
// runs out, the kernel raises the timeout flag exactly as a stalled kernel
// would, and returns: no copy or tensor-core operation is ever in flight, so
// the context stays usable and gdn_device_status() reports GDN_ERR_TIMEOUT.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace gdn {
namespace {

__global__ void wait_selftest_kernel(uint32_t polls, int *flag) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_fence_init();
  }
  __syncthreads();
  // phase 0 never completes: no thread arrives and no copy is armed on the barrier
  const bool done = tc::mbar_wait(&bar, 0, polls);
  if (!done && threadIdx.x == 0) raise_device_flag(flag, kDevTimeout);
}

}  // namespace

cudaError_t launch_wait_selftest(uint32_t polls, int *flag, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(polls, flag);
  return cudaGetLastError();
}

}  // namespace gdn
