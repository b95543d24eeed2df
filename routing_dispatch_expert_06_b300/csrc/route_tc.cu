// Router logits on the sm_103a tensor cores: s = x W_rᵀ by tcgen05 MMA into
// tensor memory, reduced over d in fp32 and written as partial logits; the
// softmax, top-k, weights and column sums run in route_select_kernel
// (route_select.cu), which reads them.
//
// [MoE 模型原理 §2.1] s_t = W_r x_t + b_r (the bias is added by the select
// kernel).
//
// Tiles of 128 tokens.  When there are few tiles (small T), nsplit CTAs share
// one tile's reduction over d: each takes a contiguous run of its segments and
// writes its own fp32 partial logits, part[split][t][e]; the select kernel
// adds the splits in split order, so the result does not depend on which CTA
// runs first.  A CTA walks units (tile, split) b, b + grid, ...  With E > 128
// and one split, clusters of two CTAs share 256-token tiles (PAIR, see the
// kernel): 170 against 176 us of routing on the d = 7168, E = 256 layer.
// Warps:
//   warp 0     TMA producer: x tile [128 × 64] and W_r tile [NP × 64] per
//              64-wide k-block, two k-blocks per stage when NP <= 64
//              (NP = E rounded up to a power of two >= 32; rows past E
//              and columns past d arrive as zeros from the copy engine's
//              out-of-bounds fill)
//   warp 1     TMEM allocator and MMA issuer: tcgen05.mma M=128, N=NP, K=16,
//              bf16 in, fp32 accumulate, into one of two TMEM buffers
//   warps 2..  epilogue, G groups of four warps (G = 2 for NP = 32, else 4):
//              one token row and NP/G columns per thread
//
// Precision.  The tensor cores' fp32 accumulation over a long K chain drifts
// (about 2e-5 relative over d = 7168, above the 1e-5 logit tolerance), so
// the reduction over d is cut into segments of kSegBlocks k-blocks (512
// elements): each segment starts a fresh accumulator, and the epilogue adds
// the segment sums into fp32 registers while the MMA fills the other buffer.
// Short chains over small partial sums keep the logits close to the exact
// dot product.  (256-element segments gave the same precision but twice the
// tensor-memory drain per k-block, which held the d = 7168, E = 256 router
// back by ~8%.)
//
// After a unit's last segment each epilogue thread stores its row's NP/G sums
// (16-byte stores; a row's columns are contiguous) while the MMA already runs
// the next unit into the other buffer.  Every wait is bounded (4 s); on a
// timeout the kernel records MOE_ERR_TIMEOUT, drains its copies and MMAs,
// frees its tensor memory and returns.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int kTileM = kRouteTileM;  // 128 tokens per tile
constexpr int kTileK = 64;           // one 128-byte swizzle row of bf16
constexpr int kSegBlocks = 8;        // k-blocks per accumulation segment (K = 512)
constexpr int kMaxStages = 8;
constexpr uint64_t kWaitLimitNs = 4000000000ull;
constexpr int kMaxNP = 256;
constexpr size_t kMinSmem = 120 * 1024;  // one CTA per SM (it may take all of TMEM)

template <int G>
constexpr int epi_threads() { return 128 * G; }

// 64-wide k-blocks per pipeline stage.  The MMA thread's fixed work per stage
// (barrier wait, commit, loop) with its 4 MMAs per k-block measured ~0.33 us
// per k-block whatever N, which paced the narrow routers (E <= 64, stages of
// 20-24 KiB); two k-blocks per stage halve that work at the same bytes in
// flight.  At NP = 256 a stage already holds 48 KiB and only 4 fit.
__host__ __device__ constexpr int route_stage_kblocks(int NP) { return NP <= 64 ? 2 : 1; }

struct RouteTcArgs {
  int64_t T;
  int d, E, NP, stages;
  uint32_t tmem_cols;
  int nsplit;        // CTAs sharing one tile's reduction over d
  float* part;       // [nsplit][T][E] fp32 partial logits (no bias)
  int32_t* status;
};

// NPG = NP / G columns per epilogue thread.  PAIR (NP = 256, one split):
// clusters of two CTAs run the 2-SM MMA (cta_group::2, M = 256 tokens,
// N = 256 experts) on 256-token tiles; each CTA stages its own 128 token rows
// and half of W_r (tmW boxes of 128 rows), the copies of both complete on the
// even CTA's barriers, the even CTA issues the MMAs and multicasts its
// commits, and each CTA drains its own 128 rows of the accumulator.  Per SM
// and k-block that is 32 KiB of operands instead of 48 KiB, so two k-blocks
// per stage fit three times.
template <int NPG, int G, bool PAIR>
__global__ void __launch_bounds__(64 + 128 * G, 1)
    route_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmW, const RouteTcArgs a) {
  constexpr int NP = G * NPG;
  constexpr int CH = 16;  // columns per tensor-memory load
  constexpr int kEpiThreads = epi_threads<G>();
  constexpr int KB = PAIR ? 2 : route_stage_kblocks(NP);
  constexpr int BROWS = PAIR ? NP / 2 : NP;     // W_r rows staged by this CTA
  constexpr int TILE = PAIR ? 2 * kTileM : kTileM;  // tokens per unit
  static_assert(!PAIR || NP == 256, "pairs only for NP = 256");
  static_assert(kSegBlocks % KB == 0, "segments hold whole stages");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
  __shared__ uint64_t tfull_bar[2], tempty_bar[2], drain_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? tc::cluster_ctarank() : 0u;  // 0 = the pair's MMA issuer
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t a_box = kTileM * kTileK * 2;
  const uint32_t b_box = uint32_t(BROWS) * kTileK * 2;
  const uint32_t a_bytes = KB * a_box;
  const uint32_t b_bytes = KB * b_box;
  uint8_t* sA = smem;
  uint8_t* sB = smem + a.stages * a_bytes;
  const int nk = (a.d + kTileK - 1) / kTileK;
  const int nseg = (nk + kSegBlocks - 1) / kSegBlocks;
  const int64_t n_tiles = (a.T + TILE - 1) / TILE;
  // Work unit u: tile u / nsplit, segments [seg_lo, seg_hi) of split u % nsplit
  // (PAIR: nsplit = 1); CTA (pair) b takes units b, b + grid, ...
  const int64_t n_units = n_tiles * a.nsplit;
  const int64_t unit0 = PAIR ? blockIdx.x / 2 : blockIdx.x;
  const int64_t unit_step = PAIR ? gridDim.x / 2 : gridDim.x;
  auto seg_range = [&](int64_t u, int& lo, int& hi) {
    const int sp = int(u % a.nsplit);
    lo = int(int64_t(sp) * nseg / a.nsplit);
    hi = int(int64_t(sp + 1) * nseg / a.nsplit);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      tc::mbar_init(&full_bar[s], 1);
      tc::mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull_bar[b], 1);
      // PAIR: one arrival per epilogue warp of both CTAs, on the even CTA's.
      tc::mbar_init(&tempty_bar[b], PAIR ? 2 * kEpiThreads / 32 : kEpiThreads);
    }
    tc::mbar_init(&drain_bar, 1);
    s_abort = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmX);
    tc::prefetch_tmap(&tmW);
  }
  // A pair allocates its tensor memory collectively, and the peer's barriers
  // must be initialised before any copy or commit of the pair signals them.
  if constexpr (PAIR) tc::cluster_sync();
  if (warp == 1) {
    if constexpr (PAIR) {
      tc::tmem_alloc_pair(&s_tmem, a.tmem_cols);
      tc::tmem_relinquish_pair();
    } else {
      tc::tmem_alloc(&s_tmem, a.tmem_cols);
      tc::tmem_relinquish();
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = s_tmem;
  volatile int* abort_flag = &s_abort;
  // The select kernel may be scheduled from now on; it waits for this grid to
  // finish and flush before reading the partial logits.
  tc::grid_launch_dependents();
  auto give_up = [&]() {
    *abort_flag = 1;
    set_status(a.status, MOE_ERR_TIMEOUT);
  };

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int64_t u = unit0; u < n_units && ok; u += unit_step) {
      const int32_t m0 = int32_t((u / a.nsplit) * TILE + int64_t(rank) * kTileM);
      int seg_lo, seg_hi;
      seg_range(u, seg_lo, seg_hi);
      const int kb_hi = min(nk, seg_hi * kSegBlocks);
      // Stage kb holds k-blocks KB·kb .. KB·kb + KB - 1; one past d (odd nk)
      // arrives as zeros.
      for (int kb = seg_lo * kSegBlocks / KB; kb * KB < kb_hi; ++kb) {
        if (!tc::mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
          give_up();
          ok = false;
          break;
        }
        if constexpr (PAIR) {
          // Both CTAs' copies complete on the even CTA's full barrier, which
          // expects the bytes of the whole pair.
          if (rank == 0) tc::mbar_arrive_expect_tx(&full_bar[stage], 2 * (a_bytes + b_bytes));
          const uint32_t bar = tc::mapa(tc::smem_u32(&full_bar[stage]), 0);
#pragma unroll
          for (int h = 0; h < KB; ++h) {
            const int kx = (kb * KB + h) * kTileK;
            tc::tma_load_2d_pair(&tmX, bar, sA + stage * a_bytes + h * a_box, kx, m0);
            tc::tma_load_2d_pair(&tmW, bar, sB + stage * b_bytes + h * b_box, kx,
                                 int(rank) * BROWS);
          }
        } else {
          tc::mbar_arrive_expect_tx(&full_bar[stage], a_bytes + b_bytes);
#pragma unroll
          for (int h = 0; h < KB; ++h) {
            const int kx = (kb * KB + h) * kTileK;
            tc::tma_load_2d(&tmX, &full_bar[stage], sA + stage * a_bytes + h * a_box, kx, m0);
            tc::tma_load_2d(&tmW, &full_bar[stage], sB + stage * b_bytes + h * b_box, kx, 0);
          }
        }
        ++issued;
        if (++stage == a.stages) stage = 0, phase ^= 1u;
      }
    }
    // Drain: the last `stages` copies this thread issued must land before the
    // CTA exits (on the normal path the MMA issuer has consumed them all).  In
    // a pair the even CTA's full barriers track the copies of both CTAs.
    if (rank == 0) {
      const int64_t first = issued > a.stages ? issued - a.stages : 0;
      for (int64_t i = first; i < issued; ++i)
        tc::mbar_wait(&full_bar[i % a.stages], uint32_t((i / a.stages) & 1), nullptr,
                      kWaitLimitNs);
    }
  } else if (warp == 1 && rank == 0) {
    // ---------------- MMA issuer (whole warp, one elected lane issues) -----
    const uint32_t idesc = tc::idesc_bf16_f32(TILE, NP);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t seg_count = 0;  // segments issued by this CTA (all tiles)
    bool ok = true;
    for (int64_t u = unit0; u < n_units && ok; u += unit_step) {
      int seg_lo, seg_hi;
      seg_range(u, seg_lo, seg_hi);
      for (int sg = seg_lo; sg < seg_hi && ok; ++sg, ++seg_count) {
        const uint32_t buf = seg_count & 1u;
        const uint32_t par = ((seg_count >> 1) & 1u) ^ 1u;
        // Waits are taken by every lane and agreed on, so the warp stays
        // converged and its operands warp-uniform.
        const bool free_acc = __all_sync(
            0xffffffffu, PAIR ? tc::mbar_wait_cluster(&tempty_bar[buf], par, abort_flag,
                                                      kWaitLimitNs)
                              : tc::mbar_wait(&tempty_bar[buf], par, abort_flag, kWaitLimitNs));
        if (!free_acc) {
          give_up();
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d_tmem = tmem_base + buf * uint32_t(NP);
        const int kb_end = min(nk, (sg + 1) * kSegBlocks);
        for (int kb = sg * kSegBlocks / KB; kb * KB < kb_end; ++kb) {
          if (!__all_sync(0xffffffffu,
                          tc::mbar_wait(&full_bar[stage], phase, abort_flag, kWaitLimitNs))) {
            give_up();
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t a0 = tc::smem_u32(sA + stage * a_bytes);
          const uint32_t b0 = tc::smem_u32(sB + stage * b_bytes);
          const bool first = kb * KB == sg * kSegBlocks;
          const uint64_t ad0 = tc::sdesc_kmajor_sw128(a0), bd0 = tc::sdesc_kmajor_sw128(b0);
#pragma unroll
          for (int j = 0; j < KB * kTileK / 16; ++j) {
            const uint32_t h = uint32_t(j / (kTileK / 16)), q = uint32_t(j % (kTileK / 16));
            const uint64_t ad = tc::sdesc_advance(ad0, h * a_box + q * 32);
            const uint64_t bd = tc::sdesc_advance(bd0, h * b_box + q * 32);
            if constexpr (PAIR)
              tc::mma_bf16_pair_w(d_tmem, ad, bd, idesc, (first && j == 0) ? 0u : 1u);
            else
              tc::mma_bf16_w(d_tmem, ad, bd, idesc, (first && j == 0) ? 0u : 1u);
          }
          if constexpr (PAIR)
            tc::mma_commit_pair_mc_w(&empty_bar[stage], 0x3);
          else
            tc::mma_commit_w(&empty_bar[stage]);
          if (++stage == a.stages) stage = 0, phase ^= 1u;
        }
        if (ok) {
          if constexpr (PAIR)
            tc::mma_commit_pair_mc_w(&tfull_bar[buf], 0x3);
          else
            tc::mma_commit_w(&tfull_bar[buf]);
        }
      }
    }
    // Drain: every MMA this warp issued completes before TMEM is freed.
    if constexpr (PAIR)
      tc::mma_commit_pair_w(&drain_bar);
    else
      tc::mma_commit_w(&drain_bar);
    tc::mbar_wait(&drain_bar, 0, nullptr, kWaitLimitNs);
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    const int quarter = warp & 3;        // TMEM lanes [32·quarter, 32·quarter + 32)
    const int g = (warp - 2) >> 2;       // column group: [g·NPG, g·NPG + NPG)
    const int row = quarter * 32 + lane;
    const int E = a.E;
    const int col0 = g * NPG;
    const int ncol = min(NPG, E - col0);
    const uint32_t t_lane = tmem_base + (uint32_t(quarter * 32) << 16) + uint32_t(col0);
    uint32_t seg_count = 0;
    bool ok = true;
    for (int64_t u = unit0; u < n_units; u += unit_step) {
      const int64_t t = (u / a.nsplit) * TILE + int64_t(rank) * kTileM + row;
      int seg_lo, seg_hi;
      seg_range(u, seg_lo, seg_hi);
      float v[NPG];
#pragma unroll
      for (int j = 0; j < NPG; ++j) v[j] = 0.f;
      for (int sg = seg_lo; sg < seg_hi; ++sg, ++seg_count) {
        const uint32_t buf = seg_count & 1u;
        if (ok) {
          // The tensor-memory loads are warp-collective: the whole warp takes
          // the same branch.
          ok = __all_sync(0xffffffffu, tc::mbar_wait(&tfull_bar[buf], (seg_count >> 1) & 1u,
                                                     abort_flag, kWaitLimitNs));
          if (!ok) give_up();
        }
        if (ok) {
          tc::fence_after_sync();
#pragma unroll
          for (int c0 = 0; c0 < NPG; c0 += CH) {
            uint32_t r[CH];
            tc::tmem_ld_x16(t_lane + buf * uint32_t(NP) + uint32_t(c0), r);
            tc::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < CH; ++j) v[c0 + j] += __uint_as_float(r[j]);
          }
          tc::fence_before_sync();
          if constexpr (PAIR) {
            // One arrival per warp on the even CTA's barrier.
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_cluster(tc::mapa(tc::smem_u32(&tempty_bar[buf]), 0));
          } else {
            tc::mbar_arrive(&tempty_bar[buf]);
          }
        }
      }
      if (ok && t < a.T && ncol > 0) {
        float* dst = a.part + (int64_t(u % a.nsplit) * a.T + t) * E + col0;
        if ((E & 3) == 0) {
#pragma unroll
          for (int j = 0; j < NPG; j += 4)
            if (j < ncol)
              __stcg(reinterpret_cast<float4*>(dst + j), make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]));
        } else {
#pragma unroll
          for (int j = 0; j < NPG; ++j)
            if (j < ncol) __stcg(dst + j, v[j]);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  // Neither CTA of a pair leaves (or frees its tensor memory) while the other
  // may still signal its barriers or feed its MMAs.
  if constexpr (PAIR) tc::cluster_sync();
  tc::fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    if constexpr (PAIR)
      tc::tmem_dealloc_pair(tmem_base, a.tmem_cols);
    else
      tc::tmem_dealloc(tmem_base, a.tmem_cols);
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

bool encode_2d(EncodeTiledFn encode, CUtensorMap* m, const void* base, int64_t inner,
               int64_t outer, uint32_t box_inner, uint32_t box_outer) {
  const cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
  const cuuint64_t strides[1] = {cuuint64_t(inner) * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <int NPG, int G, bool PAIR>
cudaError_t launch_g(const CUtensorMap& tmX, const CUtensorMap& tmW, RouteTcArgs a,
                     int64_t n_units, cudaStream_t st) {
  auto kernel = route_tc_kernel<NPG, G, PAIR>;
  const void* kp = reinterpret_cast<const void*>(kernel);
  // As many stages as fit beside the kernel's static shared memory.
  const size_t stage_bytes =
      PAIR ? size_t(2) * (size_t(kTileM) + G * NPG / 2) * kTileK * 2
           : size_t(route_stage_kblocks(G * NPG)) * (size_t(kTileM) + G * NPG) * kTileK * 2;
  const size_t budget = size_t(device_smem_optin()) - kernel_static_smem(kp) - 1024;
  int stages = int(budget / stage_bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return cudaErrorInvalidValue;
  a.stages = stages;
  size_t smem = 1024 + size_t(stages) * stage_bytes;
  if (smem < kMinSmem) smem = kMinSmem;
  cudaError_t err = ensure_dynamic_smem(kp, smem);
  if (err != cudaSuccess) return err;
  const int sms = device_sms();
  if constexpr (!PAIR) {
    const unsigned grid = unsigned(n_units < sms ? n_units : sms);
    kernel<<<grid, 64 + 128 * G, smem, st>>>(tmX, tmW, a);
    return cudaGetLastError();
  } else {
    // Persistent clusters of two: as many as can be resident, at most one per
    // unit.
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(64 + 128 * G);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.gridDim = dim3(2);
    int clusters = 0;
    err = max_active_clusters(kp, cfg, &clusters);
    if (err != cudaSuccess) return err;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    cfg.gridDim = dim3(unsigned(2 * (n_units < clusters ? n_units : clusters)));
    err = cudaLaunchKernelEx(&cfg, kernel, tmX, tmW, a);
    return err != cudaSuccess ? err : cudaGetLastError();
  }
}

}  // namespace

// Splits per tile: enough (tile, split) units to give every SM of a
// 148-SM part about one unit, at most one split per segment.  Depends on the
// configuration only, so results do not depend on the device.
int route_tc_nsplit(const moe_config_t& c) {
  const int64_t n_tiles = (c.T + kTileM - 1) / kTileM;
  const int nseg = int(((c.d + kTileK - 1) / kTileK + kSegBlocks - 1) / kSegBlocks);
  int64_t ns = kRouteSplitUnits / n_tiles;
  if (ns > nseg) ns = nseg;
  if (ns < 1) ns = 1;
  return int(ns);
}

int route_tc_np(const moe_config_t& c) {
  int NP = 32;
  while (NP < c.E) NP <<= 1;
  return NP;
}

bool route_tc_supported(const moe_config_t& c) {
  return c.dtype == MOE_DT_BF16 && c.E <= kMaxNP && c.k <= 16;
}

cudaError_t launch_route_tc(const moe_config_t& c, const void* x, const void* Wr, float* part,
                            int32_t* status, cudaStream_t st) {
  if (!route_tc_supported(c)) return cudaErrorInvalidValue;
  EncodeTiledFn encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  RouteTcArgs a{};
  a.T = c.T;
  a.d = c.d;
  a.E = c.E;
  const int NP = route_tc_np(c);
  a.NP = NP;
  a.tmem_cols = uint32_t(2 * NP);  // two accumulator buffers
  a.nsplit = route_tc_nsplit(c);
  a.part = part;
  a.status = status;

  // CTA pairs on 256-token tiles when one split covers d and E > 128.
  const bool pair = NP == 256 && a.nsplit == 1;

  CUtensorMap tmX, tmW;
  if (!encode_2d(encode, &tmX, x, c.d, c.T, kTileK, kTileM)) return cudaErrorInvalidValue;
  if (!encode_2d(encode, &tmW, Wr, c.d, c.E, kTileK, uint32_t(pair ? NP / 2 : NP)))
    return cudaErrorInvalidValue;
  const int64_t tile = pair ? 2 * kTileM : kTileM;
  const int64_t n_units = ((c.T + tile - 1) / tile) * a.nsplit;
  cudaError_t err;
  switch (NP) {
    case 32: err = launch_g<16, 2, false>(tmX, tmW, a, n_units, st); break;
    case 64: err = launch_g<16, 4, false>(tmX, tmW, a, n_units, st); break;
    case 128: err = launch_g<32, 4, false>(tmX, tmW, a, n_units, st); break;
    default:
      err = pair ? launch_g<64, 4, true>(tmX, tmW, a, n_units, st)
                 : launch_g<64, 4, false>(tmX, tmW, a, n_units, st);
      break;
  }
  count_launch();
  return err;
}

}  // namespace moe
