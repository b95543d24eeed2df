// Self-test of the bounded mbarrier wait (tc::mbar_wait) that every
// tensor-core kernel's pipeline uses: a block waits on a barrier that nothing
// signals; the wait must give up after its time limit and the kernel must
// record MOE_ERR_TIMEOUT and return, leaving the context usable.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  __syncwarp();
  // Nothing arrives on `bar`: phase 0 never completes.
  const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(&bar, 0, nullptr, limit_ns));
  if (!ok && threadIdx.x == 0) set_status(status, MOE_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(int32_t* status, uint64_t limit_ns, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
