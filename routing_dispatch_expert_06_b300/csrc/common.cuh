// Shared device helpers for the MoE-layer kernels (sm_103a).
#pragma once

#include <utility>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Tokens per dispatch chunk (one CTA of the histogram / assign kernels).
constexpr int kChunkTokens = 256;
// Tokens per CTA of the warp router (one psum partial row per CTA).
constexpr int kRouteTokensSimt = 64;
// Rows per router tile in the tensor-core router.
constexpr int kRouteTileM = 128;
// Target count of (tile, split) work units of the tensor-core router.
constexpr int64_t kRouteSplitUnits = 148;
// Largest W_r (bytes) the warp router stages in shared memory.
constexpr size_t kRouteWarpSmemMax = 96 * 1024;

// Workspace layout (byte offsets), all 256-byte aligned.
struct WsLayout {
  size_t status;        // int32 status word
  size_t chunk_counts;  // int32 [n_chunks, E]: histogram, then chunk bases in place
  size_t psum_partial;  // fp32 [n_route_blocks, E] (warp router)
  size_t route_part;    // fp32 [nsplit, T, E] partial logits (tensor-core router)
  size_t reroute;       // reroute only: int32 cand, ids1, pos0, pos1 [T, k]; kept0, counts1 [E]
  size_t combine_cnt;   // fuse_combine only: int32 [T, 2·column tiles] arrival counters
  size_t total;
  int64_t n_chunks;
  int64_t n_route_blocks;
};

// The workspace starts with a 272 KiB header that moe_workspace_init clears:
// the status word, grid-completion counters, and the router's fixed-point
// column-sum accumulators (every kernel leaves them at zero).
constexpr int kPsumReplicas = 32;       // copies of the accumulator, spread over L2
constexpr int kPsumFixedMaxE = 1024;
constexpr size_t kWsRouteCounter = 64;
constexpr size_t kWsDispatchCounter = 128;
constexpr size_t kWsDispatchBarrier = 192;  // int [2]: arrivals, departures
constexpr size_t kWsTailTiles = 256;        // int [2]: next tail tile, CTAs done
constexpr size_t kWsPsumFixed = 16384;  // uint64 [kPsumReplicas][kPsumFixedMaxE]
constexpr size_t kWsHeaderBytes =
    kWsPsumFixed + size_t(kPsumReplicas) * kPsumFixedMaxE * sizeof(unsigned long long);
// Column sums Σ_t p are kept as integers: p rounded to 31 fraction bits.
constexpr float kPsumFixScale = 2147483648.0f;  // 2^31: p <= 1 fits in 32 bits
constexpr double kPsumFixInv = 1.0 / 2147483648.0;

// Called by every thread of every block once its results are written.
// Returns true in exactly one block, the last to arrive, after which that
// block sees every other block's global writes.  The counter returns to 0,
// ready for the next launch.
__device__ __forceinline__ bool last_block_to_finish(int* counter, int* s_flag) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(counter, 1);
    const bool last = prev == int(gridDim.x) - 1;
    if (last) atomicExch(counter, 0);
    *s_flag = last;
  }
  __syncthreads();
  const bool last = *s_flag != 0;
  if (last) __threadfence();
  return last;
}

// psum[i] = Σ_b part[b][i] for b = 0, 1, ..., nblk-1 in that order (fixed,
// deterministic); threads of one block stride over i.
__device__ __forceinline__ void sum_partials_rows(int64_t nblk, int E, const float* part,
                                                  float* psum) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float s = 0.f;
    for (int64_t b = 0; b < nblk; ++b) s += __ldcg(part + b * E + e);
    psum[e] = s;
  }
}

// [MoE 模型原理 §3.2] f_i = counts_i/T, p̄_i = psum_i/T, L_aux = α·E·Σ_i f_i p̄_i,
// computed by one block of kAuxThreads threads: thread j takes experts j,
// j + kAuxThreads, ... in order, then a fixed-shape tree adds the threads'
// sums.  Explicitly rounded products and sums keep the result identical
// wherever the routine runs (the stand-alone statistics kernel, or the last
// histogram block of a forward pass).  red: kAuxThreads floats of shared memory.
constexpr int kAuxThreads = 256;
// Statistics inputs: from L2 (written by other blocks), or (SHARED) from this
// block's shared memory.
template <bool SHARED, typename V>
__device__ __forceinline__ V ld_stat(const V* p) {
  if constexpr (SHARED)
    return *p;
  else
    return __ldcg(p);
}
template <bool SHARED = false>
__device__ __forceinline__ void aux_stats_block(int E, int64_t T, float alpha,
                                                const int32_t* counts, const float* psum,
                                                float* f, float* pbar, float* l_aux, float* red) {
  const int j = threadIdx.x;
  float prod = 0.f;
  for (int e = j; e < E; e += kAuxThreads) {
    const float fi = float(ld_stat<SHARED>(counts + e)) / float(T);
    const float pi = ld_stat<SHARED>(psum + e) / float(T);
    f[e] = fi;
    pbar[e] = pi;
    prod = __fadd_rn(prod, __fmul_rn(fi, pi));
  }
  red[j] = prod;
  __syncthreads();
  for (int s = kAuxThreads / 2; s > 0; s >>= 1) {
    if (j < s) red[j] = __fadd_rn(red[j], red[j + s]);
    __syncthreads();
  }
  if (j == 0) *l_aux = __fmul_rn(__fmul_rn(alpha, float(E)), red[0]);
}

// psum[c] = (Σ over the kPsumReplicas copies of fixed[c]) / 2^31 for c < E,
// and the copies return to zero; threads of one block stride over c.  Called
// by one block after every block that added into the copies has finished.
__device__ __forceinline__ void psum_from_fixed(int E, unsigned long long* fixed, float* psum) {
  for (int c = threadIdx.x; c < E; c += blockDim.x) {
    unsigned long long fx = 0;
#pragma unroll 8
    for (int r = 0; r < kPsumReplicas; ++r) fx += __ldcg(fixed + r * kPsumFixedMaxE + c);
#pragma unroll 8
    for (int r = 0; r < kPsumReplicas; ++r) __stcg(fixed + r * kPsumFixedMaxE + c, 0ull);
    psum[c] = float(double(fx) * kPsumFixInv);
  }
}

// Sum of one value per thread over a block of kAuxThreads threads, in a fixed
// tree order (deterministic); every thread gets the result.
__device__ __forceinline__ float block_sum_fixed(float v, float* red) {
  const int j = threadIdx.x;
  red[j] = v;
  __syncthreads();
  for (int s = kAuxThreads / 2; s > 0; s >>= 1) {
    if (j < s) red[j] = __fadd_rn(red[j], red[j + s]);
    __syncthreads();
  }
  const float r = red[0];
  __syncthreads();
  return r;
}

// Routing-health indicators (one block of kAuxThreads threads), from counts
// before capacity and kept rows after it:
//   health[0] = -Σ q ln q, q_i = counts_i/(T·k)   health[1] = var(counts)
//   health[2] = var(kept)                          health[3] = 1 - Σkept/(T·k)
// (population variances over the E experts).  Σ kept is an exact integer sum.
template <bool SHARED = false>
__device__ __forceinline__ void routing_health_block(int E, int64_t T, int k,
                                                     const int32_t* counts, const int32_t* kept,
                                                     float* health, float* red,
                                                     unsigned long long* s_kept) {
  const int j = threadIdx.x;
  if (j == 0) *s_kept = 0ull;
  __syncthreads();
  const double n = double(T) * double(k);
  const float mc = float(n / double(E));
  float h = 0.f, vc = 0.f;
  unsigned long long ks = 0ull;
  for (int e = j; e < E; e += kAuxThreads) {
    const int32_t c = ld_stat<SHARED>(counts + e);
    const float q = float(double(c) / n);
    if (q > 0.f) h = __fadd_rn(h, -__fmul_rn(q, logf(q)));
    const float dc = float(c) - mc;
    vc = __fadd_rn(vc, __fmul_rn(dc, dc));
    ks += unsigned(ld_stat<SHARED>(kept + e));
  }
  atomicAdd(s_kept, ks);
  h = block_sum_fixed(h, red);
  vc = block_sum_fixed(vc, red);
  const unsigned long long kept_sum = *s_kept;
  const float mk = float(double(kept_sum) / double(E));
  float vk = 0.f;
  for (int e = j; e < E; e += kAuxThreads) {
    const float dk = float(ld_stat<SHARED>(kept + e)) - mk;
    vk = __fadd_rn(vk, __fmul_rn(dk, dk));
  }
  vk = block_sum_fixed(vk, red);
  if (j == 0) {
    health[0] = h;
    health[1] = vc / float(E);
    health[2] = vk / float(E);
    health[3] = float(1.0 - double(kept_sum) / n);
  }
}

// Aux-statistics outputs for the dispatch's last histogram block (forward
// pass only).  psum_fixed: when set, psum is first formed from the router's
// fixed-point column sums (psum_from_fixed).  health: when set, the
// routing-health indicators (routing_health_block) from counts and kept.
struct AuxArgs {
  float alpha;
  float* psum;
  float* f;
  float* pbar;
  float* l_aux;
  unsigned long long* psum_fixed;
  float* health;
  const int32_t* counts_f;  // counts for f and health when not the launch's own (reroute)
};

// Per-token row work (scatter, combine) is done by one warp per (token, part
// of the row).  With few tokens the row is cut into parts of at least
// min_part 16-byte vectors so that about kRowWorkItems warps have work (a
// handful of warps walking long rows one load round after another is
// latency-bound); with T >= kRowWorkItems a part is the whole row.
constexpr int64_t kRowWorkItems = 2048;
struct RowSplit {
  int64_t n_parts, part_vecs;
};
inline RowSplit row_split(int64_t T, int64_t row_vecs, int64_t min_part) {
  int64_t parts = (kRowWorkItems + T - 1) / T;
  const int64_t max_parts = (row_vecs + min_part - 1) / min_part;
  if (parts > max_parts) parts = max_parts;
  if (parts < 1) parts = 1;
  const int64_t pv = (row_vecs + parts - 1) / parts;
  return {(row_vecs + pv - 1) / pv, pv};
}

// Programmatic dependent launch.  A kernel launched with launch_pdl may be
// scheduled while the previous kernel in the stream is still running: it
// calls pdl_wait() before it reads or writes anything that kernel touches
// (pdl_wait returns once that kernel has completed and its writes are
// visible), then pdl_trigger(), which lets the next kernel be scheduled.
// Triggering only after the wait keeps every earlier kernel complete by the
// time any later one passes its own wait.  Without a programmatic dependency
// both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Record the first asynchronous error in the status word.
__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

// Grid-wide barrier of a cooperative launch (every block resident at once):
// each block arrives on bar[0], then waits until `expect` blocks have arrived.
// The wait is bounded: after limit_ns it records MOE_ERR_TIMEOUT and returns
// false, so a block that never arrives cannot hang the grid.  Every block
// then calls grid_barrier_depart (also after a timeout); the last to depart
// resets both counters, ready for the next launch.  s_ok: one int of shared
// memory.
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ bool grid_barrier_wait(int* bar, int expect, int32_t* status,
                                                  uint64_t limit_ns, int* s_ok) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    atomicAdd(bar, 1);
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    int ok = 1;
    while (ld_acquire_gpu(bar) < expect) {
      uint64_t t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > limit_ns) {
        ok = 0;
        set_status(status, MOE_ERR_TIMEOUT);
        break;
      }
      __nanosleep(64);
    }
    *s_ok = ok;
  }
  __syncthreads();
  __threadfence();
  return *s_ok != 0;
}
__device__ __forceinline__ void grid_barrier_depart(int* bar) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(bar + 1, 1) == int(gridDim.x) - 1) {
      atomicExch(bar, 0);
      atomicExch(bar + 1, 0);
    }
  }
}

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// σ of the expert FFN: ReLU, or GELU in its tanh form
// 0.5·u·(1 + tanh(√(2/π)·(u + 0.044715·u³))).
__device__ __forceinline__ float act_relu(float u) { return u > 0.f ? u : 0.f; }
__device__ __forceinline__ float act_gelu_tanh(float u) {
  const float k0 = 0.7978845608028654f;  // √(2/π)
  float inner = k0 * (u + 0.044715f * u * u * u);
  return 0.5f * u * (1.f + tanhf(inner));
}
__device__ __forceinline__ float apply_act(int act, float u) {
  return act == MOE_ACT_RELU ? act_relu(u) : act_gelu_tanh(u);
}

__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }

}  // namespace moe
