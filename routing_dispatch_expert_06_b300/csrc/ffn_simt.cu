// Grouped expert GEMM on CUDA cores, for fp32 layers (and as a cross-check of
// the tensor-core path for bf16).
//
// [MoE 模型原理 §1] E_i(x) = W2 σ(W1 x + b1) + b2: each expert's GEMM covers
// only that expert's rows of the dispatch buffer (the ragged groups given by
// offsets), so no padding to a fixed capacity is computed.
//
// One CTA computes a 64×64 tile of one expert; tiles never straddle two
// experts.  fp32 accumulation, 4×4 outputs per thread, operands staged in
// shared memory as fp32.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kBM = 64, kBN = 64, kBK = 16;

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(256)
    gemm_simt_kernel(int E, int N, int K, int64_t max_rows, const int32_t* __restrict__ offsets,
                     const TIn* __restrict__ A, const TIn* __restrict__ B,
                     const float* __restrict__ bias, int act, TOut* __restrict__ out) {
  __shared__ float As[kBK][kBM + 4];
  __shared__ float Bs[kBK][kBN + 4];
  __shared__ int s_e, s_m0, s_mend;
  const int tid = threadIdx.x;
  if (tid == 0) {
    // Map blockIdx.y to (expert, first row) by walking the per-expert tile counts.
    // Offsets are clamped to [0, max_rows] so no tile reaches outside A or out.
    auto clamp_row = [&](int e) {
      const int32_t v = offsets[e];
      return int32_t(v < 0 ? 0 : (int64_t(v) > max_rows ? max_rows : v));
    };
    int64_t y = blockIdx.y;
    int found = -1, m0 = 0, m_end = 0;
    for (int e = 0; e < E; ++e) {
      const int32_t a = clamp_row(e), b = clamp_row(e + 1);
      const int tiles = b > a ? (b - a + kBM - 1) / kBM : 0;
      if (y < tiles) {
        found = e;
        m0 = a + int(y) * kBM;
        m_end = b;
        break;
      }
      y -= tiles;
    }
    s_e = found;
    s_m0 = m0;
    s_mend = m_end;
  }
  __syncthreads();
  const int e = s_e;
  if (e < 0) return;
  const int m0 = s_m0;
  const int m_end = s_mend;
  const int n0 = blockIdx.x * kBN;
  const TIn* Be = B + int64_t(e) * N * K;
  const int tx = tid & 15, ty = tid >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kBK) {
    // 64×16 tiles of A and B: 1024 elements each, 4 per thread.
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + i * 256;
      const int r = idx / kBK, kk = idx % kBK;
      const int gr = m0 + r, gk = k0 + kk;
      As[kk][r] = (gr < m_end && gk < K) ? to_f32(A[int64_t(gr) * K + gk]) : 0.f;
      const int gn = n0 + r;
      Bs[kk][r] = (gn < N && gk < K) ? to_f32(Be[int64_t(gn) * K + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gr = m0 + ty * 4 + i;
    if (gr >= m_end) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= N) continue;
      float v = acc[i][j] + (bias ? bias[int64_t(e) * N + gn] : 0.f);
      if (act >= 0) v = apply_act(act, v);
      out[int64_t(gr) * N + gn] = from_f32<TOut>(v);
    }
  }
}

cudaError_t launch_gemm_simt(int dtype, int E, int N, int K, int64_t max_rows,
                             const int32_t* offsets, const void* A, const void* B,
                             const float* bias, int act, void* out, cudaStream_t st) {
  const int64_t ytiles = (max_rows + kBM - 1) / kBM + E;
  dim3 grid(unsigned((N + kBN - 1) / kBN), unsigned(ytiles));
  if (dtype == MOE_DT_F32)
    gemm_simt_kernel<float, float><<<grid, 256, 0, st>>>(
        E, N, K, max_rows, offsets, static_cast<const float*>(A), static_cast<const float*>(B), bias, act,
        static_cast<float*>(out));
  else
    gemm_simt_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, 256, 0, st>>>(
        E, N, K, max_rows, offsets, static_cast<const __nv_bfloat16*>(A),
        static_cast<const __nv_bfloat16*>(B), bias, act, static_cast<__nv_bfloat16*>(out));
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
