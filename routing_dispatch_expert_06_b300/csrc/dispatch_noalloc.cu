// moe_dispatch_noalloc: the dispatch stage with its scratch memory held in a
// fixed device array of this library instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory of their own: for example a
// plugin running inside a host framework whose memory pool owns the whole
// device, or a latency-critical path where the implicit synchronisation of
// cudaMalloc is not allowed.  They can still pass the inputs and outputs of
// the dispatch (which they hold already) but not a workspace.  This entry
// point runs the same kernels as moe_dispatch with the per-chunk histogram
// kept in g_dispatch_scratch below, and allocates nothing.
//
// Limits and sharing:
//  * scratch holds ceil(T/256) · E int32 values; at most kScratchInts
//    (262144 int32 = 1 MiB), e.g. T <= 262144 tokens at E = 256.  Larger
//    calls are rejected with MOE_ERR_INVALID_ARG before any launch.
//  * every GPU that loads the library holds the 1 MiB array until the
//    process exits.
//  * every call on a device uses the same array, which keeps the last call's
//    contents; the histogram pass overwrites every entry it later reads, so
//    nothing needs clearing between calls.  Calls that overlap on the GPU
//    (different streams without ordering between them) race on the array.
//  * the first call on each device looks up the array's device address
//    (cudaGetSymbolAddress, with that device current) and caches it; make
//    that first call before any stream capture.
#include <mutex>
#include <string>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int64_t kScratchInts = 262144;  // 1 MiB of int32
constexpr int kMaxDevices = 64;

__device__ __align__(256) int32_t g_dispatch_scratch[kScratchInts];

std::mutex g_mu;
int32_t* g_scratch_addr[kMaxDevices] = {};

// Device address of g_dispatch_scratch on the current device (looked up once
// per device).  In host code the array's name is only a host-side stand-in.
cudaError_t scratch_address(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_dispatch_noalloc(const moe_config_t* cfg, const void* x,
                                             const int32_t* topk_ids, int32_t* counts,
                                             int32_t* kept, int32_t* offsets, int32_t* slot_row,
                                             int32_t* row_token, void* xd, int32_t* status,
                                             void* stream) {
  const StageRange range("moe_dispatch_noalloc");
  // Argument checks shared with the other entry points (they set the message
  // returned by moe_last_error).
  size_t ws_bytes = 0;
  moe_status_t s = moe_workspace_size(cfg, &ws_bytes);
  if (s != MOE_OK) return s;
  if (!x || !topk_ids || !counts || !kept || !offsets || !slot_row || !row_token ||
      (!xd && !cfg->fuse_dispatch))
    return report_error(MOE_ERR_INVALID_ARG, "moe_dispatch_noalloc: NULL tensor");
  // With fuse_dispatch no row is copied (the first GEMM gathers the rows).
  if (cfg->fuse_dispatch) xd = nullptr;
  if (cfg->reroute)
    return report_error(MOE_ERR_UNSUPPORTED,
                        "moe_dispatch_noalloc: reroute needs the workspace of moe_dispatch");
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(xd) & 15))
    return report_error(MOE_ERR_INVALID_ARG,
                        "moe_dispatch_noalloc: x and xd must be 16-byte aligned");
  const int64_t n_chunks = (cfg->T + kChunkTokens - 1) / kChunkTokens;
  if (n_chunks * cfg->E > kScratchInts)
    return report_error(MOE_ERR_INVALID_ARG,
                        "moe_dispatch_noalloc: ceil(T/256)*E exceeds the fixed scratch of "
                        "262144 int32 (1 MiB); use moe_dispatch with a workspace");
  int32_t* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess)
    return report_error(MOE_ERR_CUDA, "moe_dispatch_noalloc: cudaGetSymbolAddress failed");
  const int64_t C = moe_capacity(cfg);
  e = launch_dispatch(*cfg, C, x, topk_ids, counts, kept, offsets, slot_row, row_token, xd,
                      scratch, status, nullptr, nullptr, nullptr, nullptr,
                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK
                          : report_error(MOE_ERR_CUDA, "moe_dispatch_noalloc: launch failed");
}
