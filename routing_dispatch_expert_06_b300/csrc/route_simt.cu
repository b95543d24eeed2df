// Router on CUDA cores: logits, softmax, top-k, combine weights, and per-CTA
// partial column sums of the probabilities.
//
// [MoE 模型原理 §2.1] s_t = W_r x_t + b_r, p_t = softmax(s_t);
// [MoE 模型原理 §2.2] S_t = TopK(p_t, k), p̃ = p/Σ_{S_t} p or raw p.
//
// One warp per token (groups of 8 tokens per block).  Lanes split the model
// width d; each lane keeps 32 running dot products (one per expert of the
// current 32-expert block) over its slice, then a transposing butterfly gives
// lane L the logit of expert L of the block.  Column sums of p: per warp over
// its tokens, per block over its warps (fp32, fixed order), then added as
// 64-bit fixed-point integers (exact, order-free) into the workspace's
// accumulator copies, converted by the last block (or later, by the whole
// layer's dispatch).  This is the fp32 router
// (tf32 tensor cores could not meet an fp32 logit tolerance) and it also
// serves bf16 inputs for any E; the tensor-core router covers bf16 at scale.
#include "common.cuh"
#include "kernels.h"

namespace moe {

struct Bf16x8 {
  __device__ static void unpack(const uint4& v, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 p = __bfloat1622float2(h[i]);
      f[2 * i] = p.x;
      f[2 * i + 1] = p.y;
    }
  }
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Softmax, top-k and weights for one token whose E fp32 logits sit in s_log
// (warp-private shared memory).  Adds p_{t,i} into s_ps[i].  Writes ids and
// weights for token t.  Ranking is on the fp32 logits, or with sel_bias
// (nullable) on the fp32 sums logit + sel_bias (the weights still use the
// logits); equal keys go to the lower expert index.  Destroys s_log (selected
// entries become -inf; logits are finite for finite inputs, so a taken entry
// never wins again).
__device__ __forceinline__ void softmax_topk_warp(float* s_log, float* s_ps, int E, int k,
                                                  int renorm, int64_t t, int32_t* topk_ids,
                                                  float* topk_w, const float* sel_bias,
                                                  int32_t* cand) {
  const int lane = lane_id();
  float mx = -INFINITY;
  for (int e = lane; e < E; e += 32) mx = fmaxf(mx, s_log[e]);
  mx = warp_max(mx);
  float z = 0.f;
  for (int e = lane; e < E; e += 32) z += expf(s_log[e] - mx);
  z = warp_sum(z);
  const float inv_z = 1.f / z;
  for (int e = lane; e < E; e += 32) s_ps[e] += expf(s_log[e] - mx) * inv_z;

  int my_id = -1;
  float my_p = 0.f;
  // With cand (nullable, [T,k]) the rounds continue to rank 2k - 1 (at most
  // E): the token's next candidates for an overflow reroute.
  const int rounds = cand ? min(2 * k, E) : k;
  for (int r = 0; r < rounds; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      float v = s_log[e];
      if (sel_bias) v += sel_bias[e];
      if (v > bv || (v == bv && e < bi)) {
        bv = v;
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == r) {
      my_id = bi;
      my_p = expf(s_log[bi] - mx) * inv_z;
    }
    __syncwarp();
    if (lane == (bi & 31)) s_log[bi] = -INFINITY;
    __syncwarp();
  }
  float sel = warp_sum(lane < k ? my_p : 0.f);
  if (lane < k) {
    topk_ids[t * k + lane] = my_id;
    topk_w[t * k + lane] = renorm ? my_p / sel : my_p;
  }
  if (cand && lane >= k && lane < 2 * k) cand[t * k + lane - k] = lane < rounds ? my_id : -1;
}

template <typename TIn>
__global__ void __launch_bounds__(256)
    route_simt_kernel(int64_t T, int d, int E, int k, int renorm, const TIn* __restrict__ x,
                      const TIn* __restrict__ Wr, const float* __restrict__ br, float* logits,
                      int32_t* topk_ids, float* topk_w, unsigned long long* psum_fixed,
                      float* psum, int* counter, int finish, const float* __restrict__ sel_bias,
                      int32_t* cand) {
  __shared__ int s_flag;
  extern __shared__ float smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* s_log = smem + warp * E;
  float* s_ps = smem + 8 * E + warp * E;
  for (int e = lane; e < E; e += 32) s_ps[e] = 0.f;
  // Groups of 8 tokens, one per warp: group b, b + grid, ...
  const int64_t n_groups = (T + 7) / 8;
  for (int64_t grp = blockIdx.x; grp < n_groups; grp += gridDim.x) {
    const int64_t t = grp * 8 + warp;
    if (t >= T) continue;  // warp-uniform
    const TIn* xr = x + t * d;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int ne = min(32, E - e0);
      float acc[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] = 0.f;
      for (int c = lane; c < d; c += 32) {
        const float xv = to_f32(xr[c]);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (i < ne) acc[i] = fmaf(xv, to_f32(Wr[int64_t(e0 + i) * d + c]), acc[i]);
      }
      // Transposing butterfly: at offset o the lanes with bit o set keep the
      // upper half of the values and send the lower half; after the five
      // steps lane L holds the full sum of value L (fixed order).
#pragma unroll
      for (int half = 16; half >= 1; half >>= 1) {
        const bool upper = (lane & half) != 0;
#pragma unroll
        for (int j = 0; j < half; ++j) {
          const float send = upper ? acc[j] : acc[j + half];
          const float keep = upper ? acc[j + half] : acc[j];
          acc[j] = keep + __shfl_xor_sync(0xffffffffu, send, half);
        }
      }
      if (lane < ne) s_log[e0 + lane] = acc[0] + br[e0 + lane];
    }
    __syncwarp();
    if (logits)
      for (int e = lane; e < E; e += 32) logits[t * E + e] = s_log[e];
    __syncwarp();
    softmax_topk_warp(s_log, s_ps, E, k, renorm, t, topk_ids, topk_w, sel_bias, cand);
    __syncwarp();
  }
  __syncthreads();
  // Column sums: the block's warps in order (fp32), then one fixed-point
  // atomic per column into this block's copy of the accumulator.
  unsigned long long* rep = psum_fixed + (blockIdx.x % kPsumReplicas) * kPsumFixedMaxE;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float s = 0.f;
    for (int w = 0; w < 8; ++w) s += smem[8 * E + w * E + e];
    const unsigned long long fx = __double2ull_rn(double(s) * double(kPsumFixScale));
    if (fx) atomicAdd(rep + e, fx);
  }
  if (finish && last_block_to_finish(counter, &s_flag)) psum_from_fixed(E, psum_fixed, psum);
}

// Router on CUDA cores for small expert counts (bf16, E <= 32, W_r small
// enough for shared memory): at E <= 32 the contraction has at most 32 flop
// per byte of x, so it is bound by reading x and needs no tensor cores.  One
// warp per token: lanes take 16-byte chunks of x (8 bf16), multiply them by
// the same chunk of every W_r row (staged once per CTA in shared memory) and
// keep EB running fp32 dot products.  A transposing butterfly leaves lane L
// with the full sum for expert L >> (5 - log2 EB); softmax, top-k and weights
// follow as in the other routers.  The block's column sums of p go to
// psum_partial, and the last block to finish adds the rows in order.
template <int EB>
__global__ void __launch_bounds__(256)
    route_warp_kernel(int64_t T, int d, int E, int k, int renorm,
                      const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ Wr,
                      const float* __restrict__ br, float* logits, int32_t* topk_ids,
                      float* topk_w, float* psum_partial, float* psum, int* counter,
                      const float* __restrict__ sel_bias, int32_t* cand) {
  extern __shared__ uint4 s_w[];  // [E][d/8] 16-byte chunks of W_r
  __shared__ float s_log[8][32];
  __shared__ float s_ps[8][32];
  __shared__ int s_flag;
  constexpr int kSteps = EB == 8 ? 3 : EB == 16 ? 4 : 5;  // halving steps
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nch = d / 8;
  const uint4* wg = reinterpret_cast<const uint4*>(Wr);
  for (int i = threadIdx.x; i < E * nch; i += blockDim.x) s_w[i] = wg[i];
  s_ps[warp][lane] = 0.f;
  __syncthreads();
  const int col = lane >> (5 - kSteps);
  const bool holder = (lane & ((1 << (5 - kSteps)) - 1)) == 0;
  const int64_t nwarps = int64_t(gridDim.x) * 8;
  for (int64_t t = int64_t(blockIdx.x) * 8 + warp; t < T; t += nwarps) {
    float acc[EB];
#pragma unroll
    for (int e = 0; e < EB; ++e) acc[e] = 0.f;
    const uint4* xr = reinterpret_cast<const uint4*>(x + t * d);
    for (int c = lane; c < nch; c += 32) {
      float xf[8];
      Bf16x8::unpack(__ldcs(xr + c), xf);
#pragma unroll
      for (int e = 0; e < EB; ++e) {
        if (e < E) {
          float wf[8];
          Bf16x8::unpack(s_w[e * nch + c], wf);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[e] = fmaf(xf[j], wf[j], acc[e]);
        }
      }
    }
    int n = EB;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      if (n > 1) {
        const int half = n >> 1;
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < EB / 2; ++j) {
          if (j < half) {
            const float send = upper ? acc[j] : acc[j + half];
            const float keep = upper ? acc[j + half] : acc[j];
            acc[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        n = half;
      } else {
        acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
      }
    }
    if (holder && col < E) s_log[warp][col] = acc[0] + br[col];
    __syncwarp();
    if (logits && lane < E) logits[t * E + lane] = s_log[warp][lane];
    __syncwarp();
    softmax_topk_warp(s_log[warp], s_ps[warp], E, k, renorm, t, topk_ids, topk_w, sel_bias,
                      cand);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float s = 0.f;
    for (int w2 = 0; w2 < 8; ++w2) s += s_ps[w2][e];
    psum_partial[int64_t(blockIdx.x) * E + e] = s;
  }
  if (last_block_to_finish(counter, &s_flag)) sum_partials_rows(gridDim.x, E, psum_partial, psum);
}

cudaError_t launch_route_simt(const moe_config_t& c, const void* x, const void* Wr,
                              const float* br, float* logits, int32_t* ids, float* w,
                              unsigned long long* psum_fixed, float* psum, int* counter,
                              bool finish, const float* sel_bias, int32_t* cand,
                              cudaStream_t st) {
  // Groups of 8 tokens; at most kSimtMaxBlocks blocks (a constant, so each
  // block's share of tokens depends on T only).
  constexpr int64_t kSimtMaxBlocks = 1184;
  const int64_t groups = (c.T + 7) / 8;
  const int64_t nblk = groups < kSimtMaxBlocks ? groups : kSimtMaxBlocks;
  const size_t smem = size_t(16) * c.E * sizeof(float);
  cudaError_t err;
  if (c.dtype == MOE_DT_F32) {
    err = ensure_dynamic_smem(reinterpret_cast<const void*>(route_simt_kernel<float>), smem);
    if (err != cudaSuccess) return err;
    route_simt_kernel<float><<<unsigned(nblk), 256, smem, st>>>(
        c.T, c.d, c.E, c.k, c.renormalize, static_cast<const float*>(x),
        static_cast<const float*>(Wr), br, logits, ids, w, psum_fixed, psum, counter,
        finish ? 1 : 0, sel_bias, cand);
  } else {
    err = ensure_dynamic_smem(reinterpret_cast<const void*>(route_simt_kernel<__nv_bfloat16>),
                              smem);
    if (err != cudaSuccess) return err;
    route_simt_kernel<__nv_bfloat16><<<unsigned(nblk), 256, smem, st>>>(
        c.T, c.d, c.E, c.k, c.renormalize, static_cast<const __nv_bfloat16*>(x),
        static_cast<const __nv_bfloat16*>(Wr), br, logits, ids, w, psum_fixed, psum, counter,
        finish ? 1 : 0, sel_bias, cand);
  }
  count_launch();
  return cudaGetLastError();
}

bool route_warp_supported(const moe_config_t& c) {
  return c.dtype == MOE_DT_BF16 && c.E <= 32 && size_t(c.E) * c.d * 2 <= kRouteWarpSmemMax;
}

cudaError_t launch_route_warp(const moe_config_t& c, const void* x, const void* Wr,
                              const float* br, float* logits, int32_t* ids, float* w,
                              float* psum_partial, float* psum, int* counter,
                              const float* sel_bias, int32_t* cand, cudaStream_t st) {
  if (!route_warp_supported(c)) return cudaErrorInvalidValue;
  const int sms = device_sms();
  // Blocks of 8 warps, about 8 tokens per warp, at most 4 blocks per SM; one
  // psum_partial row per block (at most ceil(T / 64) rows).
  const int64_t want = (c.T + kRouteTokensSimt - 1) / kRouteTokensSimt;
  const unsigned grid = unsigned(want < int64_t(4) * sms ? want : int64_t(4) * sms);
  const size_t smem = size_t(c.E) * c.d * 2;
  auto run = [&](auto kernel) {
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kernel), smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, 256, smem, st>>>(c.T, c.d, c.E, c.k, c.renormalize,
                                    static_cast<const __nv_bfloat16*>(x),
                                    static_cast<const __nv_bfloat16*>(Wr), br, logits, ids, w,
                                    psum_partial, psum, counter, sel_bias, cand);
    return cudaGetLastError();
  };
  cudaError_t err = c.E <= 8 ? run(route_warp_kernel<8>)
                    : c.E <= 16 ? run(route_warp_kernel<16>)
                                : run(route_warp_kernel<32>);
  count_launch();
  return err;
}

}  // namespace moe
