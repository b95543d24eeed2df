// Grouped expert GEMM for layers whose experts hold few rows (the decode
// regime: capacity C <= 64), on the sm_103a tensor cores.
//
// [MoE 模型原理 §1] E_i(x) = W2 σ(W1 x + b1) + b2, per expert over its rows of
// the dispatch buffer (offsets[e] .. offsets[e+1]):
//
//   out[row, n] = epi( Σ_k A[row, k] · B[e, n, k] + bias[e, n] )
//
// the same result as gemm_tc_kernel, with the operands' roles swapped: the
// MMA's M = 128 runs over weight rows n and its N = NT (16, 32 or 64) over
// the expert's rows, D[n, j] = Σ_k B[e, n, k] · A[offsets[e] + j, k].  With a
// handful of rows per expert the usual orientation spends almost all of its
// MMA work on 128- or 256-row tiles that are nearly empty; here each MMA is
// NT columns wide and the kernel streams the touched experts' weights.
//
// One CTA per SM, persistent over tiles (expert e with rows, 128 weight rows),
// expert-major with the weight-row tile fastest.  Warps:
//   warp 0     TMA producer: per stage two 64-wide k-blocks of
//              B[e, n0 .. n0+127, :] (2 × 16 KiB) and of A[offsets[e] .. +NT, :],
//              128-byte swizzle, a ring of as many stages as fit (6 at NT = 16)
//   warp 1     TMEM allocator and MMA issuer: tcgen05.mma.cta_group::1
//              kind::f16, M = 128, N = NT, two accumulators of NT columns
//   warps 2-5  epilogue, one per TMEM lane quarter: thread = weight row n,
//              NT columns = the expert's rows; bias, σ, bf16; for each row j
//              the warp stores 32 consecutive outputs (64 bytes)
// Two k-blocks per stage halve the issuing thread's fixed work per k-block
// (barrier wait, commit, loop): with NT = 16 its 4 MMAs cost nothing on the
// tensor pipe, and one 64-wide k-block per stage measured ~600 clocks of that
// thread's time, which held one SM to ~58 GB/s of weights.
// Rows of the A tile past the expert's end (the next expert's rows, or past
// the buffer: zero-filled by the copy engine) are computed and not stored.
// Every wait is bounded (4 s): on a timeout the kernel records
// MOE_ERR_TIMEOUT, drains its copies and MMAs, frees its tensor memory and
// returns.
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int kTileN = 128;  // weight rows per tile (MMA M)
constexpr int kTileK = 64;   // one 128-byte swizzle row of bf16
constexpr int kBoxes = 2;    // 64-wide k-blocks per stage
constexpr int kMaxStages = 12;
constexpr int kEpiWarp0 = 2;
constexpr int kEpiWarps = 4;
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr uint64_t kWaitLimitNs = 4000000000ull;
constexpr int kMaxExperts = 1024;
constexpr int kMaxSwapRows = 64;  // largest NT

template <int ACT>
__device__ __forceinline__ float epi_act(float u) {
  if constexpr (ACT == MOE_ACT_RELU) return u > 0.f ? u : 0.f;
  if constexpr (ACT == MOE_ACT_GELU_TANH)
    return 0.5f * u * (1.f + tc::tanh_fast(0.7978845608028654f * (u + 0.044715f * u * u * u)));
  return u;
}

// expert_max: only experts holding 1 .. expert_max rows are computed (the
// others are left to the regular kernel); every expert with rows when it is
// at least NT.  Each tile's MMA is as wide as its expert's rows rounded up to
// 16 (at most NT), so a 3-row expert costs a 16-wide MMA.
template <int ACT, int NT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_swap_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, int E, int N, int K,
                     const int32_t* __restrict__ offsets, const float* __restrict__ bias,
                     __nv_bfloat16* __restrict__ out, int64_t max_rows, int32_t* status,
                     int stages, int expert_max) {
  constexpr uint32_t kTmemCols = 2 * NT < 32 ? 32 : 2 * NT;  // two accumulators
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
  __shared__ uint64_t tfull_bar[2], tempty_bar[2], drain_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_tp[kMaxExperts + 1];      // experts with rows before e (prefix)
  __shared__ int32_t s_off[kMaxExperts + 1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  constexpr uint32_t b_box = kTileN * kTileK * 2;  // weight box (16 KiB)
  constexpr uint32_t a_box = NT * kTileK * 2;      // rows box
  const uint32_t b_bytes = kBoxes * b_box;
  const uint32_t a_bytes = kBoxes * a_box;
  uint8_t* sB = smem;
  uint8_t* sA = smem + stages * b_bytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      tc::mbar_init(&full_bar[s], 1);
      tc::mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&tfull_bar[a], 1);
      tc::mbar_init(&tempty_bar[a], kEpiWarps);
    }
    tc::mbar_init(&drain_bar, 1);
    s_abort = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmA);
    tc::prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tc::tmem_alloc(&s_tmem, kTmemCols);
    tc::tmem_relinquish();
  }
  // Launched with programmatic dependent launch, so the grid may start while
  // the previous kernel (the scatter, or the first GEMM) still runs.  The A
  // rows come from that kernel and are read only after griddepcontrol.wait.
  // offsets comes from a kernel before it, and every kernel of the layer
  // waits for its own predecessor before it lets the next one start, so
  // offsets is complete once this grid runs: the tile list, and (when every
  // CTA has a tile) the first stages' weight copies, go ahead of the wait.
  // Prefix over experts with 1 .. expert_max rows: warp 0 scans runs of
  // experts, one run per lane.  Offsets are clamped to [0, max_rows] and read
  // from L2 (no stale L1 line from an earlier launch).
  if (warp == 0) {
    auto clamp_row = [&](int e) {
      const int32_t v = __ldcg(offsets + e);
      return int32_t(v < 0 ? 0 : (int64_t(v) > max_rows ? max_rows : v));
    };
    const int per = (E + 31) / 32;
    const int lo = lane * per, hi = min(E, lo + per);
    int run = 0;
    auto takes = [&](int32_t a, int32_t b) { return b > a && b - a <= expert_max; };
    for (int e = lo; e < hi; ++e) {
      const int32_t a = clamp_row(e), b = clamp_row(e + 1);
      s_off[e] = a;
      run += takes(a, b) ? 1 : 0;
    }
    if (lane == 31) s_off[E] = clamp_row(E);
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    int acc = incl - run;
    for (int e = lo; e < hi; ++e) {
      s_tp[e] = acc;
      acc += takes(clamp_row(e), clamp_row(e + 1)) ? 1 : 0;
    }
    if (lane == 31) s_tp[E] = incl;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = s_tmem;

  const int n_tn = (N + kTileN - 1) / kTileN;
  const int64_t total = int64_t(s_tp[E]) * n_tn;
  const int nk = (K + kBoxes * kTileK - 1) / (kBoxes * kTileK);  // stages per tile
  volatile int* abort_flag = &s_abort;
  // Early weight copies only when every CTA has a tile.  With fewer tiles
  // than CTAs (T = 1 on the E = 64 layer: 66 and 96 tiles) they measured
  // slower, in either GEMM (the first one's own run took 9.7 -> 12.3 us in
  // the kernel timeline); the cause is not known, so such grids wait first.
  const bool early_w = total >= int64_t(gridDim.x);
  if (!early_w) {
    tc::grid_dependency_wait();
    tc::grid_launch_dependents();
  }
  auto give_up = [&]() {
    *abort_flag = 1;
    set_status(status, MOE_ERR_TIMEOUT);
  };
  // Tile i: the (i / n_tn)-th expert with rows, weight rows (i % n_tn)·128.
  auto tile_expert = [&](int64_t i, int& e, int& n0) {
    const int p = int(i / n_tn);
    int lo = 0, hi = E;  // s_tp[lo] <= p < s_tp[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_tp[mid] <= p)
        lo = mid;
      else
        hi = mid;
    }
    e = lo;
    n0 = int(i % n_tn) * kTileN;
  };

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    // The weight boxes of the first `stages` stages are issued before the
    // previous kernel has finished (weights are inputs; each stage's full
    // barrier already expects its A boxes too, so it cannot complete early).
    int pre = 0;
    if (early_w) {
      int64_t i = blockIdx.x;
      int kb = 0;
      for (; pre < stages && i < total; ++pre) {
        int e, n0;
        tile_expert(i, e, n0);
        tc::mbar_arrive_expect_tx(&full_bar[pre], a_bytes + b_bytes);
#pragma unroll
        for (int h = 0; h < kBoxes; ++h)
          tc::tma_load_3d(&tmB, &full_bar[pre], sB + pre * b_bytes + h * b_box,
                          (kb * kBoxes + h) * kTileK, n0, e);
        if (++kb == nk) kb = 0, i += gridDim.x;
      }
    }
    if (early_w) {
      tc::grid_dependency_wait();
      tc::grid_launch_dependents();
    }
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int64_t i = blockIdx.x; i < total && ok; i += gridDim.x) {
      int e, n0;
      tile_expert(i, e, n0);
      for (int kb = 0; kb < nk; ++kb) {
        const bool early = issued < pre;  // weights already on their way
        if (!early) {
          if (!tc::mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
            give_up();
            ok = false;
            break;
          }
          // A second box past K (K/64 odd) reads zeros, which add nothing.
          tc::mbar_arrive_expect_tx(&full_bar[stage], a_bytes + b_bytes);
        }
#pragma unroll
        for (int h = 0; h < kBoxes; ++h) {
          const int kx = (kb * kBoxes + h) * kTileK;
          if (!early)
            tc::tma_load_3d(&tmB, &full_bar[stage], sB + stage * b_bytes + h * b_box, kx, n0, e);
          tc::tma_load_2d(&tmA, &full_bar[stage], sA + stage * a_bytes + h * a_box, kx,
                          s_off[e]);
        }
        ++issued;
        if (++stage == stages) stage = 0, phase ^= 1u;
      }
    }
    // Drain: the last `stages` copies must land before the CTA exits.
    const int64_t first = issued > stages ? issued - stages : 0;
    for (int64_t j = first; j < issued; ++j)
      tc::mbar_wait(&full_bar[j % stages], uint32_t((j / stages) & 1), nullptr, kWaitLimitNs);
  } else if (warp == 1) {
    // ---------------- MMA issuer (whole warp, one elected lane issues) -----
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int64_t i = blockIdx.x; i < total && ok; i += gridDim.x) {
      // Waits are taken by every lane and agreed on, so the warp stays
      // converged and its operands warp-uniform.
      if (!__all_sync(0xffffffffu,
                      tc::mbar_wait(&tempty_bar[acc], acc_phase ^ 1u, abort_flag, kWaitLimitNs))) {
        give_up();
        break;
      }
      tc::fence_after_sync();
      const uint32_t d_tmem = tmem_base + uint32_t(acc * NT);
      int e, n0;
      tile_expert(i, e, n0);
      const int rows = s_off[e + 1] - s_off[e];
      const int n_mma = rows >= NT ? NT : ((rows + 15) / 16) * 16;
      const uint32_t idesc = tc::idesc_bf16_f32(kTileN, n_mma < 16 ? 16 : n_mma);
      for (int kb = 0; kb < nk; ++kb) {
        if (!__all_sync(0xffffffffu,
                        tc::mbar_wait(&full_bar[stage], phase, abort_flag, kWaitLimitNs))) {
          give_up();
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t b0 = tc::smem_u32(sB + stage * b_bytes);
        const uint32_t a0 = tc::smem_u32(sA + stage * a_bytes);
        const uint64_t bd0 = tc::sdesc_kmajor_sw128(b0), ad0 = tc::sdesc_kmajor_sw128(a0);
#pragma unroll
        for (int j = 0; j < kBoxes * kTileK / 16; ++j) {
          const uint32_t h = uint32_t(j / (kTileK / 16)), q = uint32_t(j % (kTileK / 16));
          tc::mma_bf16_w(d_tmem, tc::sdesc_advance(bd0, h * b_box + q * 32),
                       tc::sdesc_advance(ad0, h * a_box + q * 32), idesc, (kb | j) != 0);
        }
        tc::mma_commit_w(&empty_bar[stage]);
        if (++stage == stages) stage = 0, phase ^= 1u;
      }
      if (!ok) break;
      tc::mma_commit_w(&tfull_bar[acc]);
      if (++acc == 2) acc = 0, acc_phase ^= 1u;
    }
    // Drain: every MMA this warp issued completes before TMEM is freed.
    tc::mma_commit_w(&drain_bar);
    tc::mbar_wait(&drain_bar, 0, nullptr, kWaitLimitNs);
  } else if (warp >= kEpiWarp0) {
    // ---------------- epilogue ----------------
    const int quarter = warp & 3;  // TMEM lanes [32·quarter, 32·quarter + 32)
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int64_t i = blockIdx.x; i < total; i += gridDim.x) {
      int e, n0;
      tile_expert(i, e, n0);
      // The tensor-memory loads are warp-collective: the whole warp takes the
      // same branch.
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&tfull_bar[acc], acc_phase, abort_flag,
                                                 kWaitLimitNs))) {
        give_up();
        break;
      }
      tc::fence_after_sync();
      const int n = n0 + quarter * 32 + lane;
      const bool valid_n = n < N;
      const float b = valid_n ? __ldg(bias + int64_t(e) * N + n) : 0.f;
      const int32_t m0 = s_off[e];
      const int rows = min(NT, s_off[e + 1] - m0);
      const uint32_t t_lane = tmem_base + (uint32_t(quarter * 32) << 16) + uint32_t(acc * NT);
#pragma unroll
      for (int c0 = 0; c0 < NT; c0 += 16) {
        if (c0 >= rows) break;  // columns past the expert's rows were not computed
        uint32_t r[16];
        tc::tmem_ld_x16(t_lane + uint32_t(c0), r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c0 + j < rows && valid_n)
            out[int64_t(m0 + c0 + j) * N + n] =
                __float2bfloat16_rn(epi_act<ACT>(__uint_as_float(r[j]) + b));
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty_bar[acc]);
      if (++acc == 2) acc = 0, acc_phase ^= 1u;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tc::tmem_dealloc(tmem_base, kTmemCols);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

template <int ACT, int NT>
cudaError_t launch_nt(const CUtensorMap& tmA, const CUtensorMap& tmB, int E, int N, int K,
                      const int32_t* offsets, const float* bias, void* out, int64_t max_rows,
                      int32_t* status, int expert_max, int grid, cudaStream_t st) {
  auto kernel = gemm_swap_kernel<ACT, NT>;
  const void* kp = reinterpret_cast<const void*>(kernel);
  const size_t stage_bytes = size_t(kBoxes) * (size_t(kTileN) + NT) * kTileK * 2;
  const size_t budget = size_t(device_smem_optin()) - kernel_static_smem(kp) - 1024;
  int stages = int(budget / stage_bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return cudaErrorInvalidValue;
  const size_t smem = 1024 + size_t(stages) * stage_bytes;
  cudaError_t err = ensure_dynamic_smem(kp, smem);
  if (err != cudaSuccess) return err;
  err = launch_pdl(kernel, dim3(unsigned(grid)), dim3(kThreads), smem, st, tmA, tmB, E, N, K,
                   offsets, bias, static_cast<__nv_bfloat16*>(out), max_rows, status, stages,
                   expert_max);
  return err != cudaSuccess ? err : cudaGetLastError();
}

template <int NT>
cudaError_t launch_act(int act, const CUtensorMap& tmA, const CUtensorMap& tmB, int E, int N,
                       int K, const int32_t* offsets, const float* bias, void* out,
                       int64_t max_rows, int32_t* status, int expert_max, int grid,
                       cudaStream_t st) {
  switch (act) {
    case MOE_ACT_RELU:
      return launch_nt<MOE_ACT_RELU, NT>(tmA, tmB, E, N, K, offsets, bias, out, max_rows, status,
                                         expert_max, grid, st);
    case MOE_ACT_GELU_TANH:
      return launch_nt<MOE_ACT_GELU_TANH, NT>(tmA, tmB, E, N, K, offsets, bias, out, max_rows,
                                              status, expert_max, grid, st);
    default:
      return launch_nt<-1, NT>(tmA, tmB, E, N, K, offsets, bias, out, max_rows, status,
                               expert_max, grid, st);
  }
}

// Tensor maps of the swapped kernel: NT-row boxes over A [max_rows, K],
// 128-row boxes over B [E, N, K].
bool encode_maps(CUtensorMap* tmA, CUtensorMap* tmB, int E, int N, int K, int64_t max_rows,
                 const void* A, const void* B, int NT) {
  EncodeTiledFn encode = get_encode();
  if (!encode) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  {
    const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(max_rows)};
    const cuuint64_t strides[1] = {cuuint64_t(K) * 2};
    const cuuint32_t box[2] = {kTileK, cuuint32_t(NT)};
    if (encode(tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(A), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  const cuuint64_t dims[3] = {cuuint64_t(K), cuuint64_t(N), cuuint64_t(E)};
  const cuuint64_t strides[2] = {cuuint64_t(K) * 2, cuuint64_t(N) * K * 2};
  const cuuint32_t box[3] = {kTileK, kTileN, 1};
  return encode(tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(B), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Rows per expert up to which the swapped kernel runs (MOE_FFN_SWAP=0 turns
// it off, a cross-check in tests).
bool gemm_swap_applies(int64_t rows_per_expert_max) {
  const char* v = std::getenv("MOE_FFN_SWAP");
  if (v && std::strcmp(v, "0") == 0) return false;
  return rows_per_expert_max >= 1 && rows_per_expert_max <= kMaxSwapRows;
}

cudaError_t launch_gemm_swap(int E, int N, int K, int64_t max_rows, int64_t rows_per_expert_max,
                             const int32_t* offsets, const void* A, const void* B,
                             const float* bias, int act, void* out, int32_t* status,
                             cudaStream_t st) {
  if (E > kMaxExperts || rows_per_expert_max < 1 || rows_per_expert_max > kMaxSwapRows)
    return cudaErrorInvalidValue;
  const int NT = rows_per_expert_max <= 16 ? 16 : rows_per_expert_max <= 32 ? 32 : 64;
  CUtensorMap tmA, tmB;
  if (!encode_maps(&tmA, &tmB, E, N, K, max_rows, A, B, NT)) return cudaErrorInvalidValue;
  const int grid = device_sms();
  const int all = int(rows_per_expert_max);
  cudaError_t err;
  if (NT == 16)
    err = launch_act<16>(act, tmA, tmB, E, N, K, offsets, bias, out, max_rows, status, all, grid,
                         st);
  else if (NT == 32)
    err = launch_act<32>(act, tmA, tmB, E, N, K, offsets, bias, out, max_rows, status, all, grid,
                         st);
  else
    err = launch_act<64>(act, tmA, tmB, E, N, K, offsets, bias, out, max_rows, status, all, grid,
                         st);
  count_launch();
  return err;
}

}  // namespace moe
