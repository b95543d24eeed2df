// Combine and load statistics.
//
// [MoE 模型原理 §2.2] y_t = Σ_{i∈S_t} p̃_{t,i} E_i(x_t); [MoE 模型原理 §5] the
// expert outputs return to token order and are merged with the routing
// weights.  Dropped slots contribute nothing and the kept weights are not
// renormalised; a token with every slot dropped gets 0 (the caller adds the
// residual).  One warp per token, 16-byte vectors, fp32 sums in rank order —
// no atomics, so the result is deterministic.
//
// [MoE 模型原理 §3.2] f_i = counts_i/T, p̄_i = Σ_t p_{t,i}/T,
// L_aux = α·E·Σ_i f_i p̄_i.
#include "common.cuh"
#include "kernels.h"

namespace moe {

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void unpack(const uint4& v, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 p = __bfloat1622float2(h[i]);
      f[2 * i] = p.x;
      f[2 * i + 1] = p.y;
    }
  }
  __device__ static uint4 pack(const float* f) {
    uint4 v;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return v;
  }
};
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ static uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

// One warp per token.  Lane r < k fetches slot r's row and weight; every
// lane then holds all k (row, weight) pairs.  Each lane takes two 16-byte
// column vectors per step and issues the 2·k row loads together before any
// arithmetic, so it keeps up to 2·KMAX independent loads in flight (one
// vector per step measured 20-25% slower on the larger layers); the weighted
// sum then runs in rank order (a dropped slot adds 0·0, which leaves the fp32
// sum unchanged).
template <typename T, int KMAX>
__global__ void __launch_bounds__(256)
    combine_kernel(int64_t n_tok, int k, int64_t row_vecs, int64_t n_parts, int64_t part_vecs,
                   int64_t max_rows, const uint4* __restrict__ yd,
                   const int32_t* __restrict__ slot_row, const float* __restrict__ w,
                   uint4* __restrict__ y) {
  constexpr int NV = Vec<T>::N;
  const int lane = threadIdx.x & 31;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  pdl_wait();
  pdl_trigger();
  for (int64_t it = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       it < n_tok * n_parts; it += warps) {
    const int64_t t = it / n_parts;
    const int64_t vb = (it % n_parts) * part_vecs;
    const int64_t ve = vb + part_vecs < row_vecs ? vb + part_vecs : row_vecs;
    int32_t my_row = lane < k ? slot_row[t * k + lane] : -1;
    if (my_row >= max_rows) my_row = -1;
    const float my_w = lane < k ? w[t * k + lane] : 0.f;
    const uint4* src[KMAX];
    float wts[KMAX];
    bool kept[KMAX];
#pragma unroll
    for (int r = 0; r < KMAX; ++r) {
      const int32_t row = __shfl_sync(0xffffffffu, my_row, r);
      kept[r] = r < k && row >= 0;
      wts[r] = kept[r] ? __shfl_sync(0xffffffffu, my_w, r) : 0.f;
      src[r] = yd + (kept[r] ? int64_t(row) * row_vecs : 0);
    }
    for (int64_t v0 = vb + lane; v0 < ve; v0 += 64) {
      uint4 buf[2][KMAX];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int r = 0; r < KMAX; ++r)
          if (kept[r] && v0 + 32 * u < ve) buf[u][r] = __ldcs(src[r] + v0 + 32 * u);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int64_t v = v0 + 32 * u;
        if (v >= ve) break;
        float acc[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) acc[i] = 0.f;
#pragma unroll
        for (int r = 0; r < KMAX; ++r) {
          float f[NV];
          if (kept[r]) {
            Vec<T>::unpack(buf[u][r], f);
          } else {
#pragma unroll
            for (int i = 0; i < NV; ++i) f[i] = 0.f;
          }
#pragma unroll
          for (int i = 0; i < NV; ++i) acc[i] = fmaf(wts[r], f[i], acc[i]);
        }
        __stcs(y + t * row_vecs + v, Vec<T>::pack(acc));
      }
    }
  }
}

// One block computes f, p̄ and L_aux (see aux_stats_block).
__global__ void __launch_bounds__(kAuxThreads)
    aux_kernel(int E, int64_t T, float alpha, const int32_t* __restrict__ counts,
               const float* __restrict__ psum, float* f, float* pbar, float* l_aux) {
  __shared__ float red[kAuxThreads];
  aux_stats_block(E, T, alpha, counts, psum, f, pbar, l_aux, red);
}

// One block computes the routing-health indicators (routing_health_block).
__global__ void __launch_bounds__(kAuxThreads)
    health_kernel(int E, int64_t T, int k, const int32_t* __restrict__ counts,
                  const int32_t* __restrict__ kept, float* health) {
  __shared__ float red[kAuxThreads];
  __shared__ unsigned long long s_kept;
  routing_health_block(E, T, k, counts, kept, health, red, &s_kept);
}

cudaError_t launch_health(const moe_config_t& c, const int32_t* counts, const int32_t* kept,
                          float* health, cudaStream_t st) {
  health_kernel<<<1, kAuxThreads, 0, st>>>(c.E, c.T, c.k, counts, kept, health);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_combine(const moe_config_t& c, int64_t max_rows, const void* yd,
                           const int32_t* slot_row, const float* w, void* y, cudaStream_t st) {
  const int elem = c.dtype == MOE_DT_BF16 ? 2 : 4;
  const int64_t row_vecs = int64_t(c.d) * elem / 16;
  const RowSplit rs = row_split(c.T, row_vecs, 64);
  const int sms = device_sms();
  const int64_t want = (c.T * rs.n_parts + 7) / 8;
  const unsigned grid = unsigned(want < int64_t(sms) * 8 ? want : int64_t(sms) * 8);
  cudaError_t err = cudaSuccess;
  auto run = [&](auto kernel) {
    err = launch_pdl(kernel, dim3(grid), dim3(256), 0, st, c.T, c.k, row_vecs, rs.n_parts,
                     rs.part_vecs, max_rows, static_cast<const uint4*>(yd), slot_row, w,
                     static_cast<uint4*>(y));
  };
  if (c.dtype == MOE_DT_BF16) {
    if (c.k <= 2) run(combine_kernel<__nv_bfloat16, 2>);
    else if (c.k <= 4) run(combine_kernel<__nv_bfloat16, 4>);
    else if (c.k <= 8) run(combine_kernel<__nv_bfloat16, 8>);
    else run(combine_kernel<__nv_bfloat16, 16>);
  } else {
    if (c.k <= 2) run(combine_kernel<float, 2>);
    else if (c.k <= 4) run(combine_kernel<float, 4>);
    else if (c.k <= 8) run(combine_kernel<float, 8>);
    else run(combine_kernel<float, 16>);
  }
  count_launch();
  return err != cudaSuccess ? err : cudaGetLastError();
}

cudaError_t launch_aux(const moe_config_t& c, const int32_t* counts, const float* psum,
                       float alpha, float* f, float* pbar, float* l_aux, cudaStream_t st) {
  aux_kernel<<<1, kAuxThreads, 0, st>>>(c.E, c.T, alpha, counts, psum, f, pbar, l_aux);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
