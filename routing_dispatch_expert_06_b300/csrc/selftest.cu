// Self-tests of the bounded waits: the mbarrier wait (tc::mbar_wait) that
// every tensor-core kernel's pipeline uses, where a block waits on a barrier
// that nothing signals, and the grid barrier of the one-pass dispatch
// (grid_barrier_wait), where the blocks wait for one block more than the grid
// holds.  Each wait must give up after its time limit, record MOE_ERR_TIMEOUT
// and return, leaving the context usable.
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

// A cooperative grid waits for gridDim.x + 1 arrivals, which never come; the
// last block to depart still resets the barrier's counters.
__global__ void __launch_bounds__(32)
    grid_barrier_timeout_kernel(int* bar, int32_t* status, uint64_t limit_ns) {
  __shared__ int s_ok;
  grid_barrier_wait(bar, int(gridDim.x) + 1, status, limit_ns, &s_ok);
  grid_barrier_depart(bar);
}

}  // namespace

cudaError_t launch_grid_barrier_timeout_selftest(int* bar, int32_t* status, uint64_t limit_ns,
                                                 cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(32);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, grid_barrier_timeout_kernel, bar, status, limit_ns);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(int32_t* status, uint64_t limit_ns, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
