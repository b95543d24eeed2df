// Router on CUDA cores: logits, softmax, top-k, combine weights, and per-CTA
// partial column sums of the probabilities.
//
// [MoE 模型原理 §2.1] s_t = W_r x_t + b_r, p_t = softmax(s_t);
// [MoE 模型原理 §2.2] S_t = TopK(p_t, k), p̃ = p/Σ_{S_t} p or raw p.
//
// One warp per token.  Lanes split the model width d; each lane keeps 32
// running dot products (one per expert of the current 32-expert block) over
// its slice, then a butterfly sum gives the logits.  This is the fp32 router
// (tf32 tensor cores could not meet an fp32 logit tolerance) and it also
// serves bf16 inputs for any E; the tensor-core router covers bf16 at scale.
#include "common.cuh"
#include "kernels.h"

namespace moe {

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
// weights for token t.  Ranking is on the fp32 logits; equal logits go to the
// lower expert index.  Destroys s_log (selected entries become -inf; logits
// are finite for finite inputs, so a taken entry never wins again).
__device__ __forceinline__ void softmax_topk_warp(float* s_log, float* s_ps, int E, int k,
                                                  int renorm, int64_t t, int32_t* topk_ids,
                                                  float* topk_w) {
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
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      float v = s_log[e];
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
      my_p = expf(bv - mx) * inv_z;
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
}

template <typename TIn>
__global__ void __launch_bounds__(256)
    route_simt_kernel(int64_t T, int d, int E, int k, int renorm, const TIn* __restrict__ x,
                      const TIn* __restrict__ Wr, const float* __restrict__ br, float* logits,
                      int32_t* topk_ids, float* topk_w, float* psum_partial) {
  extern __shared__ float smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* s_log = smem + warp * E;
  float* s_ps = smem + 8 * E + warp * E;
  for (int e = lane; e < E; e += 32) s_ps[e] = 0.f;
  const int64_t t0 = int64_t(blockIdx.x) * kRouteTokensSimt;
  for (int j = warp; j < kRouteTokensSimt; j += 8) {
    const int64_t t = t0 + j;
    if (t >= T) break;
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
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float v = warp_sum(acc[i]);
        if (lane == i && i < ne) s_log[e0 + i] = v + br[e0 + i];
      }
    }
    __syncwarp();
    if (logits)
      for (int e = lane; e < E; e += 32) logits[t * E + e] = s_log[e];
    __syncwarp();
    softmax_topk_warp(s_log, s_ps, E, k, renorm, t, topk_ids, topk_w);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float s = 0.f;
    for (int w = 0; w < 8; ++w) s += smem[8 * E + w * E + e];
    psum_partial[int64_t(blockIdx.x) * E + e] = s;
  }
}

// psum[i] = Σ_b partial[b][i], b ascending (fixed order, deterministic).
__global__ void psum_reduce_kernel(int64_t nblk, int E, const float* __restrict__ part,
                                   float* __restrict__ psum) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  float s = 0.f;
  int64_t b = 0;
  for (; b + 4 <= nblk; b += 4) {
    float a0 = part[(b + 0) * E + e], a1 = part[(b + 1) * E + e];
    float a2 = part[(b + 2) * E + e], a3 = part[(b + 3) * E + e];
    s += a0;
    s += a1;
    s += a2;
    s += a3;
  }
  for (; b < nblk; ++b) s += part[b * E + e];
  psum[e] = s;
}

cudaError_t launch_route_simt(const moe_config_t& c, const void* x, const void* Wr,
                              const float* br, float* logits, int32_t* ids, float* w,
                              float* psum_partial, float* psum, cudaStream_t st) {
  const int64_t nblk = (c.T + kRouteTokensSimt - 1) / kRouteTokensSimt;
  const size_t smem = size_t(16) * c.E * sizeof(float);
  cudaError_t err;
  if (c.dtype == MOE_DT_F32) {
    err = cudaFuncSetAttribute(route_simt_kernel<float>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (err != cudaSuccess) return err;
    route_simt_kernel<float><<<unsigned(nblk), 256, smem, st>>>(
        c.T, c.d, c.E, c.k, c.renormalize, static_cast<const float*>(x),
        static_cast<const float*>(Wr), br, logits, ids, w, psum_partial);
  } else {
    err = cudaFuncSetAttribute(route_simt_kernel<__nv_bfloat16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (err != cudaSuccess) return err;
    route_simt_kernel<__nv_bfloat16><<<unsigned(nblk), 256, smem, st>>>(
        c.T, c.d, c.E, c.k, c.renormalize, static_cast<const __nv_bfloat16*>(x),
        static_cast<const __nv_bfloat16*>(Wr), br, logits, ids, w, psum_partial);
  }
  count_launch();
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  return launch_psum_reduce(nblk, c.E, psum_partial, psum, st);
}

cudaError_t launch_psum_reduce(int64_t nblk, int E, const float* psum_partial, float* psum,
                               cudaStream_t st) {
  psum_reduce_kernel<<<unsigned((E + 255) / 256), 256, 0, st>>>(nblk, E, psum_partial, psum);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
