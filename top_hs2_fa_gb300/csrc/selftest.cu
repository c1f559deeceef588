// selftest.cu — exercises the device-side timeout path without faulting the GPU.
//
// Every wait on an mbarrier in this library is bounded (tc::mbar_wait reads %globaltimer and
// gives up after a limit), after which a kernel sets HS2_DEV_TIMEOUT in the caller's error
// word and finishes. hs2_selftest_wait_timeout launches one small CTA that waits, through that
// same helper and with a short caller-given limit, on an mbarrier nothing ever arrives on, so a
// test can check that the wait gives up, the flag is set and the context stays usable.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace hs2 {

__global__ void wait_selftest_kernel(int32_t* dev_err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  // nothing arrives on the barrier, so its phase 0 never completes
  const bool done = tc::mbar_wait(&bar, 0, limit_ns);
  if (!__all_sync(0xffffffffu, done) && threadIdx.x == 0) flag_error(dev_err, HS2_DEV_TIMEOUT);
}

cudaError_t launch_wait_selftest(int32_t* dev_err, unsigned long long limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(dev_err, limit_ns);
  return cudaGetLastError();
}

}  // namespace hs2
