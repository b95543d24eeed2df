// Softmax, top-k, combine weights and probability column sums from the fp32
// partial logits that route_tc_kernel writes.
//
// [MoE 模型原理 §2.1] s_t = W_r x_t + b_r, p_t = softmax(s_t);
// [MoE 模型原理 §2.2] S_t = TopK(p_t, k), p̃ = p/Σ_{S_t} p (or raw p);
// [MoE 模型原理 §3.2] the column sums Σ_t p_{t,i} feed p̄_i.
//
// One token per lane segment (8, 16 or 32 lanes as E <= 8, 16 or more;
// lane L holds the contiguous columns [L·EPL, L·EPL + EPL), EPL = E/32 rounded
// up to a power of two, so a lower lane holds lower expert indices).  A block
// of eight warps takes groups of tokens (group b, b + grid, ...); WPR (1, 2, 4
// or 8, from nsplit) warps share a token's split sum: each adds its own run of
// splits in split order, and the token's first warp adds the runs in order
// (a fixed association for a given T and d) and finishes the token:
//   s = Σ part + b_r, M = max s, Z = Σ exp(s - M) (segment butterflies);
//   top-k by k rounds of a warp argmax: the largest remaining value, then the
//   lowest column holding it (ties go to the lower expert index); the winner
//   is masked out and lane r of the segment keeps rank r;
//   weights exp(s - M)/Σ_{S_t} exp(s - M) (renormalised) or exp(s - M)/Z.
// Column sums Σ_t p: each token's p is rounded to fixed point with 31
// fraction bits and added as a 64-bit integer, per lane, then per block, then
// by one atomic per column into one of 32 copies of the accumulator (copies
// spread the atomics over L2).  Integer sums are exact, so Σ_t p does not
// depend on how tokens are spread over blocks or on the order in which blocks
// finish.  With `finish` set the last block to finish adds the copies,
// converts the sum to fp32 and clears them; otherwise a later kernel does
// (psum_from_fixed, in the dispatch's histogram when the whole layer runs).
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int kSelWarps = 8;


struct SelectArgs {
  int64_t T;
  int E, k, renorm, nsplit;
  int wpr;                         // warps per token (1, 2, 4, 8)
  int finish;                      // 1: the last block converts the column sums
  const float* part;               // [nsplit][T][E]
  const float* br;                 // [E]
  const float* sel_bias;           // [E] ranking-only bias, or NULL
  float* logits;                   // [T][E] or NULL
  int32_t* ids;                    // [T][k]
  int32_t* cand;                   // [T][k] experts ranked k .. 2k-1 (-1 past E), or NULL
  float* w;                        // [T][k]
  unsigned long long* psum_fixed;  // [kPsumReplicas][kPsumFixedMaxE], zero on entry and exit
  float* psum;                     // [E]
  int* counter;                    // grid-completion counter, zero on entry and on exit
};

// EPL consecutive floats at p (columns c0.. of a row); columns >= E read as
// `fill`.  VEC: E is a multiple of 4 (EPL >= 4) or of 2 (EPL == 2), so the
// row and the lane's columns are 16- (8-) byte aligned.
template <int EPL, bool VEC>
__device__ __forceinline__ void load_cols(const float* p, int c0, int E, float fill, float* v) {
  if constexpr (VEC && EPL >= 4) {
    if (c0 < E) {
#pragma unroll
      for (int j = 0; j < EPL; j += 4) {
        const float4 q = __ldcg(reinterpret_cast<const float4*>(p + c0 + j));
        v[j] = q.x, v[j + 1] = q.y, v[j + 2] = q.z, v[j + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < EPL; ++j) v[j] = fill;
    }
  } else if constexpr (VEC && EPL == 2) {
    if (c0 < E) {
      const float2 q = __ldcg(reinterpret_cast<const float2*>(p + c0));
      v[0] = q.x, v[1] = q.y;
    } else {
      v[0] = v[1] = fill;
    }
  } else {
#pragma unroll
    for (int j = 0; j < EPL; ++j) v[j] = c0 + j < E ? __ldcg(p + c0 + j) : fill;
  }
}

// Sum over the LPR lanes of a segment (xor butterfly: every lane of the
// segment ends with the same bits, since each step adds the same two
// operands in both lanes of a pair and fp addition is commutative).
template <int LPR>
__device__ __forceinline__ float seg_sum(float v) {
#pragma unroll
  for (int o = LPR / 2; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
template <int LPR>
__device__ __forceinline__ float seg_max(float v) {
#pragma unroll
  for (int o = LPR / 2; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block epilogue: s_col[c] holds this block's fixed-point column sums; one
// atomic per column into the block's copy of the accumulator, then (finish)
// the last block to finish adds the copies, converts to fp32 and clears them.
__device__ __forceinline__ void finish_column_sums(const SelectArgs& a,
                                                   const unsigned long long* s_col,
                                                   int* s_last) {
  unsigned long long* rep = a.psum_fixed + (blockIdx.x % kPsumReplicas) * kPsumFixedMaxE;
  for (int c = threadIdx.x; c < a.E; c += blockDim.x)
    if (s_col[c]) atomicAdd(rep + c, s_col[c]);
  // Every other block's atomics are complete and visible to the last block.
  if (a.finish && last_block_to_finish(a.counter, s_last))
    psum_from_fixed(a.E, a.psum_fixed, a.psum);
}

// Order-preserving map between non-NaN floats and int32 (signed compare).
__device__ __forceinline__ int ordered_key(float f) {
  const int b = __float_as_int(f);
  return b ^ ((b >> 31) & 0x7fffffff);
}
__device__ __forceinline__ float ordered_float(int key) {
  return __int_as_float(key ^ ((key >> 31) & 0x7fffffff));
}

// LPR lanes per token (8 or 16 for E <= 8 or 16, else 32), EPL columns per
// lane (LPR < 32 only with EPL = 1).  SELB: experts are ranked by the fp32
// sum logit + sel_bias (the weights still use the logit).
template <int EPL, int LPR, bool VEC, bool SELB>
__global__ void __launch_bounds__(kSelWarps * 32)
    route_select_kernel(const SelectArgs a) {
  constexpr int RPW = 32 / LPR;  // tokens per warp at a time
  __shared__ float s_bias[LPR * EPL];
  __shared__ float s_sel[SELB ? LPR * EPL : 1];
  __shared__ float s_run[kSelWarps][32 * EPL];
  __shared__ unsigned long long s_acc[kSelWarps][32 * EPL];
  __shared__ unsigned long long s_col[32 * EPL];
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane % LPR, seg = lane / LPR;
  const int E = a.E, k = a.k;
  const int c0 = sub * EPL;
  const int wpr = a.wpr, slot = warp / wpr, q = warp % wpr;
  const int rows_per_group = (kSelWarps / wpr) * RPW;
  const int64_t n_groups = (a.T + rows_per_group - 1) / rows_per_group;
  for (int c = threadIdx.x; c < LPR * EPL; c += blockDim.x) {
    s_bias[c] = c < E ? a.br[c] : 0.f;
    if constexpr (SELB) s_sel[c] = c < E ? a.sel_bias[c] : 0.f;
  }
  // Per-column fixed-point sums of p over this lane's tokens.
  unsigned long long acc[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) acc[j] = 0ull;
  __syncthreads();
  // The partial logits come from the preceding router grid.
  tc::grid_dependency_wait();
  tc::grid_launch_dependents();

  // Groups of rows_per_group tokens: group b, b + grid, ...; in a group, slot
  // `slot` takes tokens slot·RPW .. slot·RPW + RPW - 1, one per lane segment.
  for (int64_t grp = blockIdx.x; grp < n_groups; grp += gridDim.x) {
    const int64_t t = grp * rows_per_group + slot * RPW + seg;
    const bool has_row = t < a.T;

    // This warp's run of splits [s_lo, s_hi), added in split order.
    float v[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) v[j] = 0.f;
    if (has_row) {
      const int s_lo = int(int64_t(q) * a.nsplit / wpr);
      const int s_hi = int(int64_t(q + 1) * a.nsplit / wpr);
      const int64_t split_stride = a.T * E;
      const float* base = a.part + t * E;
      load_cols<EPL, VEC>(base + s_lo * split_stride, c0, E, 0.f, v);
#pragma unroll 4
      for (int s = s_lo + 1; s < s_hi; ++s) {
        float u[EPL];
        load_cols<EPL, VEC>(base + s * split_stride, c0, E, 0.f, u);
#pragma unroll
        for (int j = 0; j < EPL; ++j) v[j] += u[j];
      }
    }
    if (wpr > 1) {
#pragma unroll
      for (int j = 0; j < EPL; ++j) s_run[warp][lane * EPL + j] = v[j];
      __syncthreads();
      if (q == 0) {
#pragma unroll
        for (int j = 0; j < EPL; ++j)
          for (int r = 1; r < wpr; ++r) v[j] += s_run[warp + r][lane * EPL + j];
      }
      __syncthreads();  // s_run is reused by the next group
    }
    if (q != 0) continue;  // warp-uniform

    // Logits; a segment without a token works on zeros (no stores).
    float lmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      v[j] = c0 + j < E ? v[j] + s_bias[c0 + j] : -INFINITY;
      lmax = fmaxf(lmax, v[j]);
    }
    if (a.logits && has_row) {
      float* lrow = a.logits + t * E;
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if (c0 + j < E) lrow[c0 + j] = v[j];
    }
    const float M = seg_max<LPR>(lmax);
    float pr[EPL], z = 0.f;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      pr[j] = c0 + j < E ? __expf(v[j] - M) : 0.f;
      z += pr[j];
    }
    const float inv_z = __fdividef(1.f, seg_sum<LPR>(z));

    // Top-k by segment argmax rounds on the ranking keys (the logits, or
    // logit + sel_bias); `key` is the working copy.  my_v: the winner's logit.
    float key[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      if constexpr (SELB)
        key[j] = c0 + j < E ? v[j] + s_sel[c0 + j] : -INFINITY;
      else
        key[j] = v[j];
    }
    float my_v = -INFINITY;
    int my_i = 0;
    // With candidates the rounds continue to rank 2k - 1 (at most E).
    const int rounds = a.cand ? min(2 * k, E) : k;
    for (int r = 0; r < rounds; ++r) {
      float lm = key[0];
#pragma unroll
      for (int j = 1; j < EPL; ++j) lm = fmaxf(lm, key[j]);
      if constexpr (LPR == 32) {
        // Largest remaining key (a warp reduction on an order-preserving
        // integer image of the float), then the lowest column holding it.
        const int gkey = __reduce_max_sync(0xffffffffu, ordered_key(lm));
        const float gm = ordered_float(gkey);
        int cand = 0x7fffffff;
#pragma unroll
        for (int j = EPL - 1; j >= 0; --j)
          if (key[j] == gm) cand = c0 + j;
        const int idx = __reduce_min_sync(0xffffffffu, cand);
        float won = -INFINITY;  // the winner's logit, in the lane holding it
#pragma unroll
        for (int j = 0; j < EPL; ++j)
          if (c0 + j == idx) key[j] = -INFINITY, won = v[j];
        float wv = gm;
        if constexpr (SELB) wv = ordered_float(__reduce_max_sync(0xffffffffu, ordered_key(won)));
        if (sub == r) my_v = wv, my_i = idx;
      } else {
        const float gm = seg_max<LPR>(lm);
        unsigned bits = __ballot_sync(0xffffffffu, lm == gm);
        bits = (bits >> (seg * LPR)) & ((1u << LPR) - 1u);
        const int L = seg * LPR + __ffs(bits) - 1;
        // EPL == 1 here: lane L's only column.
        const int idx = __shfl_sync(0xffffffffu, c0, L);
        const float wv = SELB ? __shfl_sync(0xffffffffu, v[0], L) : gm;
        if (lane == L) key[0] = -INFINITY;
        if (sub == r) my_v = wv, my_i = idx;
      }
    }
    const float ev = sub < k ? __expf(my_v - M) : 0.f;
    const float inv = a.renorm ? __fdividef(1.f, seg_sum<LPR>(ev)) : inv_z;
    if (has_row && sub < k) {
      a.ids[t * k + sub] = my_i;
      a.w[t * k + sub] = ev * inv;
    }
    if (a.cand && has_row && sub >= k && sub < 2 * k)
      a.cand[t * k + sub - k] = sub < rounds ? my_i : -1;
    if (has_row) {
#pragma unroll
      for (int j = 0; j < EPL; ++j) acc[j] += __float2uint_rn(pr[j] * inv_z * kPsumFixScale);
    }
  }

  // Column sums: the block's lanes, then the common epilogue.
  if (q == 0) {
#pragma unroll
    for (int j = 0; j < EPL; ++j) s_acc[slot][lane * EPL + j] = acc[j];
  }
  __syncthreads();
  const int n_slots = kSelWarps / wpr;
  for (int c = threadIdx.x; c < E; c += blockDim.x) {
    unsigned long long fx = 0;
    for (int sl = 0; sl < n_slots; ++sl)
#pragma unroll
      for (int sg = 0; sg < RPW; ++sg) fx += s_acc[sl][sg * LPR * EPL + c];
    s_col[c] = fx;
  }
  __syncthreads();
  finish_column_sums(a, s_col, &s_last);
}

template <int EPL, int LPR, bool SELB>
cudaError_t launch_epl(const SelectArgs& a, cudaStream_t st) {
  const bool vec = EPL >= 4 ? (a.E & 3) == 0 : EPL == 2 ? (a.E & 1) == 0 : false;
  cudaLaunchConfig_t cfg{};
  const int rows_per_group = (kSelWarps / a.wpr) * (32 / LPR);
  const int64_t n_groups = (a.T + rows_per_group - 1) / rows_per_group;
  // One wave of resident blocks (the column sums do not depend on the grid).
  auto kernel = vec ? route_select_kernel<EPL, LPR, true, SELB>
                    : route_select_kernel<EPL, LPR, false, SELB>;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kSelWarps * 32, 0) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t max_blocks = int64_t(per_sm) * device_sms();
  cfg.gridDim = dim3(unsigned(n_groups < max_blocks ? n_groups : max_blocks));
  cfg.blockDim = dim3(kSelWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  // Programmatic dependent launch: the grid may be scheduled while the
  // router finishes; griddepcontrol.wait orders its reads after it.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace

cudaError_t launch_route_select(const moe_config_t& c, const float* part, int nsplit,
                                const float* br, float* logits, int32_t* ids, float* w,
                                unsigned long long* psum_fixed, float* psum, int* counter,
                                bool finish, const float* sel_bias, int32_t* cand,
                                cudaStream_t st) {
  if (c.E > 256) return cudaErrorInvalidValue;
  SelectArgs a{};
  a.T = c.T;
  a.E = c.E;
  a.k = c.k;
  a.renorm = c.renormalize;
  a.nsplit = nsplit;
  // Warps per token: about four splits per warp, at most eight warps.
  a.wpr = nsplit <= 4 ? 1 : nsplit <= 8 ? 2 : nsplit <= 16 ? 4 : 8;
  a.part = part;
  a.br = br;
  a.sel_bias = sel_bias;
  a.logits = logits;
  a.ids = ids;
  a.cand = cand;
  a.w = w;
  a.psum_fixed = psum_fixed;
  a.psum = psum;
  a.counter = counter;
  a.finish = finish ? 1 : 0;
  cudaError_t err;
  auto run = [&](auto selb) {
    constexpr bool S = decltype(selb)::value;
    if (c.E <= 8) return launch_epl<1, 8, S>(a, st);
    if (c.E <= 16) return launch_epl<1, 16, S>(a, st);
    if (c.E <= 32) return launch_epl<1, 32, S>(a, st);
    if (c.E <= 64) return launch_epl<2, 32, S>(a, st);
    if (c.E <= 128) return launch_epl<4, 32, S>(a, st);
    return launch_epl<8, 32, S>(a, st);
  };
  err = sel_bias ? run(std::true_type{}) : run(std::false_type{});
  count_launch();
  return err;
}

}  // namespace moe
