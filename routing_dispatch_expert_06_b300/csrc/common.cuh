// Shared device helpers for the MoE-layer kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Tokens per dispatch chunk (one CTA of the histogram / assign kernels).
constexpr int kChunkTokens = 256;
// Tokens per router CTA in the SIMT router (one psum partial row per CTA).
constexpr int kRouteTokensSimt = 64;
// Rows per router tile in the tensor-core router.
constexpr int kRouteTileM = 128;

// Workspace layout (byte offsets), all 256-byte aligned.
struct WsLayout {
  size_t status;        // int32 status word
  size_t chunk_counts;  // int32 [n_chunks, E]: histogram, then chunk bases in place
  size_t psum_partial;  // fp32 [n_route_blocks, E]
  size_t total;
  int64_t n_chunks;
  int64_t n_route_blocks;
};

// Record the first asynchronous error in the status word.
__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
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
