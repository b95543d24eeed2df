// Internal launchers of the MoE-layer kernels (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "moe.h"

namespace moe {

// Counts every kernel launch the library makes (reported by moe_launch_count).
void count_launch();

// Records msg as the calling thread's moe_last_error() text; returns code.
moe_status_t report_error(moe_status_t code, const char* msg);

// An NVTX range named after a library call, open for the call's lifetime, so
// a profiler's timeline shows each stage (and moe_forward's stages nested in
// it) by name.  Opened before the argument checks.  Without a tool attached
// each push and pop is one test of a null function pointer.
struct StageRange {
  explicit StageRange(const char* name);
  ~StageRange();
  StageRange(const StageRange&) = delete;
  StageRange& operator=(const StageRange&) = delete;
};

// Host-side launch helpers that query the driver once per device (or per
// kernel) and then answer from a cache, so a stage call costs little more
// than its launches.
int device_sms();                      // SMs of the current device
int device_smem_optin();               // opt-in shared memory per block
size_t kernel_static_smem(const void* kernel);
// Raise the kernel's dynamic shared-memory limit to at least `bytes` on the
// current device (once per device and size).
cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes);
// Resident clusters of the kernel for this launch shape (cached).
cudaError_t max_active_clusters(const void* kernel, const cudaLaunchConfig_t& cfg, int* clusters);

// Router on CUDA cores (fp32 or bf16, any E): logits, softmax, top-k,
// weights; per-block column sums of p in psum_partial, summed into psum by the
// last block to finish (counter: a zeroed int in the workspace).
// sel_bias (every router, nullable): rank experts by the fp32 sum
// logit + sel_bias; weights, Σp and logits stay those of the logits.
// cand (every router, nullable, [T,k]): the experts ranked k .. 2k-1 by the
// same keys (-1 past E), the next candidates of an overflow reroute.
// Σp through the fixed-point accumulator copies psum_fixed; finish: the last
// block converts them into psum (else psum_from_fixed must run later).
cudaError_t launch_route_simt(const moe_config_t& c, const void* x, const void* Wr,
                              const float* br, float* logits, int32_t* ids, float* w,
                              unsigned long long* psum_fixed, float* psum, int* counter,
                              bool finish, const float* sel_bias, int32_t* cand,
                              cudaStream_t st);

// Router on CUDA cores for bf16 layers with E <= 32 and W_r small enough for
// shared memory: one warp per token, 16-byte loads, same outputs.
bool route_warp_supported(const moe_config_t& c);
cudaError_t launch_route_warp(const moe_config_t& c, const void* x, const void* Wr,
                              const float* br, float* logits, int32_t* ids, float* w,
                              float* psum_partial, float* psum, int* counter,
                              const float* sel_bias, int32_t* cand, cudaStream_t st);

// Router logits on the tcgen05 tensor cores (bf16, E <= 256), followed by
// route_select_kernel for softmax, top-k, weights and Σp.  When T is small,
// nsplit CTAs share a 128-token tile's reduction over d, each writing its own
// partial logits.
bool route_tc_supported(const moe_config_t& c);
int route_tc_nsplit(const moe_config_t& c);
int route_tc_np(const moe_config_t& c);
// Partial router logits part[split][t][e] = Σ_{d in split} x[t,d]·W_r[e,d]
// (fp32, no bias), nsplit = route_tc_nsplit(c) splits.
cudaError_t launch_route_tc(const moe_config_t& c, const void* x, const void* Wr, float* part,
                            int32_t* status, cudaStream_t st);
// Softmax, top-k, weights, optional logits and Σ_t p from the partial logits
// (E <= 256); programmatic dependent launch after launch_route_tc.  finish:
// the last block writes psum from the fixed-point sums (else psum_from_fixed
// must run later, before psum_fixed is used again).
cudaError_t launch_route_select(const moe_config_t& c, const float* part, int nsplit,
                                const float* br, float* logits, int32_t* ids, float* w,
                                unsigned long long* psum_fixed, float* psum, int* counter,
                                bool finish, const float* sel_bias, int32_t* cand,
                                cudaStream_t st);
// One block waits on an mbarrier nothing signals, gives up after limit_ns and
// records MOE_ERR_TIMEOUT in *status (self-test of the bounded waits).
cudaError_t launch_wait_timeout_selftest(int32_t* status, uint64_t limit_ns, cudaStream_t st);
cudaError_t launch_grid_barrier_timeout_selftest(int* bar, int32_t* status, uint64_t limit_ns,
                                                 cudaStream_t st);
// One block: the routing-health indicators from counts and kept.
cudaError_t launch_health(const moe_config_t& c, const int32_t* counts, const int32_t* kept,
                          float* health, cudaStream_t st);

// Workspace buffers of an overflow reroute: cand [T,k] (the router's next
// candidates), ids1, pos0, pos1 [T,k]; kept0, counts1 [E].
struct RerouteBufs {
  const int32_t* cand;
  int32_t* ids1;
  int32_t* pos0;
  int32_t* pos1;
  int32_t* kept0;
  int32_t* counts1;
};

// Dispatch: histogram per chunk, per-expert scan + capacity, positions, row
// copy.  counter: a zeroed int for the histogram's grid-completion count (the
// last histogram block then runs the scan, and with aux != NULL also the
// f / p̄ / L_aux statistics), or NULL for a separate scan kernel.  rr (needs
// counter): the reroute variant (first fill as positions, offers, second
// fill into the room left, final rows).  xd == NULL: positions and row_token
// only, no row copy (the first GEMM then gathers its rows).  grid_bar: two
// zeroed ints for the one-pass kernel's grid barrier (T > 256 without reroute,
// when the whole grid fits on the device at once), or NULL.
cudaError_t launch_dispatch(const moe_config_t& c, int64_t C, const void* x,
                            const int32_t* ids, int32_t* counts, int32_t* kept,
                            int32_t* offsets, int32_t* slot_row, int32_t* row_token, void* xd,
                            int32_t* chunk_counts, int32_t* status, int* counter, int* grid_bar,
                            const AuxArgs* aux, const RerouteBufs* rr, cudaStream_t st);

// Grouped GEMM on CUDA cores over ragged expert row ranges (fp32 or bf16):
//   out[rows of e] = epi(A[rows of e] · B[e]ᵀ + bias[e]),  A [R,K], B [E,N,K].
// act < 0: no activation.  max_rows bounds the rows (R).
cudaError_t launch_gemm_simt(int dtype, int E, int N, int K, int64_t max_rows,
                             const int32_t* offsets, const void* A, const void* B,
                             const float* bias, int act, void* out, cudaStream_t st);

// Grouped GEMM on the tcgen05 tensor cores (bf16 in, fp32 accumulate, bf16 out).
cudaError_t launch_gemm_tc(int E, int N, int K, int64_t max_rows, const int32_t* offsets,
                           const void* A, const void* B, const float* bias, int act,
                           void* out, int32_t* status, cudaStream_t st);
// The same GEMM with its A rows gathered from the token matrix x [T, K]:
// A[row] = x[row_token[row]] (the dispatch buffer is never written).  act must
// be an activation (the first GEMM).
cudaError_t launch_gemm_tc_gather(int E, int N, int K, int64_t max_rows, const int32_t* offsets,
                                  const void* x, int64_t T, const int32_t* row_token,
                                  const void* B, const float* bias, int act, void* out,
                                  int32_t* status, cudaStream_t st);
// The second GEMM with the combine folded into its epilogue:
// yd[rows of e] = H W2[e]ᵀ + b2[e] as launch_gemm_tc, and
// y[t] = Σ_r w[t,r]·yd[slot_row[t,r]] (kept slots, rank order, fp32; 0 if none)
// by the last epilogue warp to finish a row of token t, per column range.
// cnt: 2·ceil(N / gemm_tc_bn(N)) ints per token, zero on entry (left zero).
int gemm_tc_bn(int N);
cudaError_t launch_gemm_tc_combine(int E, int N, int K, int64_t max_rows, const int32_t* offsets,
                                   const void* A, const void* B, const float* bias, void* yd,
                                   int64_t T, int k, const int32_t* row_token,
                                   const int32_t* slot_row, const float* w, void* y, int* cnt,
                                   int32_t* status, cudaStream_t st);
// The same GEMM with the operands' roles swapped (MMA M over weight rows, N
// over an expert's rows), for layers where no expert holds more than
// rows_per_expert_max <= 64 rows (gemm_swap_applies).
bool gemm_swap_applies(int64_t rows_per_expert_max);
cudaError_t launch_gemm_swap(int E, int N, int K, int64_t max_rows, int64_t rows_per_expert_max,
                             const int32_t* offsets, const void* A, const void* B,
                             const float* bias, int act, void* out, int32_t* status,
                             cudaStream_t st);

// Combine: y[t] = Σ_r w[t,r]·yd[slot_row[t,r]] (kept slots, rank order, fp32).
// Rows outside [0, max_rows) are treated as dropped.
cudaError_t launch_combine(const moe_config_t& c, int64_t max_rows, const void* yd,
                           const int32_t* slot_row, const float* w, void* y, cudaStream_t st);

// f, p̄, L_aux from counts and psum.
cudaError_t launch_aux(const moe_config_t& c, const int32_t* counts, const float* psum,
                       float alpha, float* f, float* pbar, float* l_aux, cudaStream_t st);

}  // namespace moe
