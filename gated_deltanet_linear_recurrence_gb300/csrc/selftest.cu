// selftest.cu — gdn_selftest_wait_timeout: runs the library's bounded
// mbarrier wait (tc::mbar_wait, the wait every tensor-core kernel here uses
// for its hand-offs) against a barrier that nothing completes, so that the
// failure path can be tested on a GPU without a fault or a hang: the wait
// gives up after its deadline, the kernel records GDN_ERR_DEVICE_TIMEOUT in
// the device error word and returns, and the context stays usable (contract
// in include/gdn.h).
#include <cuda_runtime.h>
#include <stdint.h>

#include "params.h"
#include "rows.cuh"
#include "tc.cuh"

namespace gdn {
namespace {

__global__ void __launch_bounds__(32, 1) selftest_wait_kernel(uint64_t timeout_ns, int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);  // one arrival expected; none ever comes
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0, timeout_ns)) raise_error(err, kErrDeviceTimeout);
}

}  // namespace

cudaError_t launch_selftest_wait(uint64_t timeout_ns, int* err, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(timeout_ns, err);
  return cudaGetLastError();
}

}  // namespace gdn
