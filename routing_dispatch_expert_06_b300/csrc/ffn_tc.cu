// Grouped expert GEMM on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// [MoE 模型原理 §1] E_i(x) = W2 σ(W1 x + b1) + b2; the experts' GEMMs run as
// one grouped GEMM over the ragged row ranges of the dispatch buffer
// (offsets[e] .. offsets[e+1]), so only kept rows are computed — no padding
// to a fixed capacity ([MoE 模型原理 §8.4]).
//
//   out[rows of e, n] = epi( Σ_k A[row, k] · B[e, n, k] + bias[e, n] )
//   A [R, K] bf16 (K contiguous), B [E, N, K] bf16 (K contiguous),
//   epi = σ then round to bf16 (first GEMM) or round to bf16 (second GEMM).
//
// Design: a persistent kernel, one CTA per SM, 10 warps.  Two variants share
// the code (template parameter PAIR):
//
//   PAIR = true (default): CTA pairs (clusters of 2) run the 2-SM MMA,
//     tcgen05.mma.cta_group::2 with M = 256: each CTA stages its own 128 A
//     rows and half of the BN-column B tile, and each SM's tensor core reads
//     A from its own shared memory and B from both.  Per SM and k-block that
//     is 16 KiB of A plus BN/2 rows of B instead of the whole B tile, which
//     halves the shared-memory traffic for B (the 1-SM variant needs about
//     192 B/clk of operand reads plus TMA writes per SM at full MMA rate, more
//     than shared memory delivers) and leaves room for 6 stages at BN = 256.
//   PAIR = false: one CTA per tile, tcgen05.mma.cta_group::1, M = 128.
//
// With many experts (E >= kTailSplitMinExperts) a GEMM is two launches: CTA
// pairs take each expert's whole 256-row tiles (and a last one holding more
// than 128 rows), and one-CTA tiles take the 1..128 rows left at the end of
// an expert.  A pair tile whose upper half lies past the expert's end spends
// half of its MMA work on rows that are not stored (1.31x the kept rows on the
// E = 256 layer, against 1.15x for 128-row tiles).  The tail launch uses
// programmatic dependent launch: it may start as soon as the pair launch is
// running, its CTAs take the SMs that pair CTAs leave, and it waits for the
// pair launch before it completes.
//
//   warp 0     TMA producer: 128×64 A tile + (BN or BN/2)×64 B tile per
//              64-wide k-block, two k-blocks per stage in a pair (one for the
//              one-CTA and gathering kernels; see stage_kblocks),
//              128-byte swizzle, a ring of as many stages as fit (GATHER:
//              the whole warp gathers the A rows, four per lane, by TMA
//              gather4 from the token matrix)
//   warp 1     TMEM allocator and (in the even CTA of a pair) MMA issuer:
//              tcgen05.mma K=16, fp32 accumulators in tensor memory, two
//              accumulator buffers so the epilogue of one tile overlaps the
//              main loop of the next
//   warps 2-9  epilogue, two warps per TMEM lane quarter (one per column
//              half): tcgen05.ld 32 columns of one row per thread, bias
//              (16-byte broadcast loads), σ, bf16, then a transpose through a
//              2 KiB per-warp shared buffer so each store instruction writes
//              8 rows × 64 contiguous bytes; rows past the expert's end and
//              columns past N are masked
// Tiles never straddle two experts.  Tile order is expert-major, and within
// an expert m-fastest, so a wave of CTAs shares the weight tile B[e, n-tile]
// through L2 while the expert's A rows stay L2-resident across n-tiles.
// Every wait is bounded: on a timeout the kernel records MOE_ERR_TIMEOUT,
// drains its own copies and MMAs, frees its tensor memory and returns.
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int kTileM = 128;             // rows per CTA (a pair covers 256)
constexpr int kTileK = 64;              // 64 bf16 = one 128-byte swizzle row
constexpr int kMaxStages = 8;
constexpr int kEpiWarp0 = 2;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
// The gathering producer runs in kGatherWarps warps (warp 0 and the warps
// after the epilogue): one warp issuing the 32 gather4 copies of every stage
// was the limit.  Warp g serves one k-block half of one pipeline stage (stage
// g / KB, half g % KB) and nothing else, so a warp waits for a stage's release
// only after it issued that stage's previous use itself: the barrier is then
// at most one phase behind and its parity wait cannot mistake an older phase
// for the one awaited.  The launch keeps stages·KB <= kGatherWarps.
constexpr int kGatherWarps = 6;
constexpr int threads_for(bool gather) {
  return 32 * (kEpiWarp0 + kEpiWarps + (gather ? kGatherWarps - 1 : 0));
}
constexpr int kEpiBufBytes = 32 * 64;   // per epilogue warp: 32 rows × 32 bf16
constexpr uint32_t kTmemCols = 512;
constexpr int kAccCols = 256;           // each of the two accumulators owns 256 columns
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s
constexpr int kMaxExperts = 1024;
// Experts from which a GEMM splits each expert's 1..128-row tail off to
// one-CTA tiles.  Measured: with E = 256 the split saves 9% of the GEMM time;
// with E = 8 or 64 the few long-K tail tiles land on the critical path and
// it cost 3-15%.
constexpr int kTailSplitMinExperts = 128;
// SMs the pair launch leaves to the tail launch when the GEMM is split and
// the tail set has at least two tiles for each of them (decided on the
// device from offsets).  The tail tiles mostly stream weights (experts with
// at most 128 rows) while the pair tiles are bound by the tensor pipe, so the
// tail launch's CTAs on these SMs start with the pair launch (programmatic
// dependent launch) and overlap the two; its remaining CTAs join as pair
// CTAs finish, taking tiles from a shared counter.
constexpr int kTailEarlySms = 28;
constexpr int kTileQueue = 4;  // dynamic tail tiles published ahead of use
enum { kActNone = -1 };

// 64-wide k-blocks per pipeline stage.  The MMA thread's fixed work per
// stage (the barrier wait, the commit, the loop) plus its 4 MMAs per k-block
// measured ~640 clocks per k-block with one k-block per stage, more than the
// ~560 clocks a 256 × 256 × 64 pair MMA keeps the tensor pipe busy, so the
// pair kernel stages two k-blocks (64 KiB per CTA, 3 stages).  The one-CTA
// kernel (96 KiB per two k-blocks: only 2 stages would fit) keeps one, and so
// does the gathering kernel, whose copies, not its MMA thread, set the pace
// (two k-blocks per stage measured 4-8% slower there).
__host__ __device__ constexpr int stage_kblocks(bool pair, bool gather) {
  return pair && !gather ? 2 : 1;
}

struct TileCoord {
  int e, m0, m_end, n0;
};

// Which of an expert's row tiles a launch covers.
enum TileSet {
  kAllTiles = 0,    // every 128-row tile (one CTA) or 256-row tile (a pair)
  kPairBody = 1,    // pairs: whole 256-row tiles, and a last one with > 128 rows
  kTail = 2,        // one CTA: the expert's last rows when 1..128 remain after
                    // its whole 256-row tiles
};

// Row tiles of an expert with `rows` rows in the given set (rows_per_tile:
// 128 for one CTA, 256 for a pair).
__device__ __forceinline__ int tiles_in_set(int rows, int set, int rows_per_tile) {
  if (rows <= 0) return 0;
  if (set == kPairBody) return rows / 256 + (rows % 256 > 128 ? 1 : 0);
  if (set == kTail) return (rows % 256 != 0 && rows % 256 <= 128) ? 1 : 0;
  return (rows + rows_per_tile - 1) / rows_per_tile;
}

// Tile i of the expert-major order.  rows_per_tile = 128 (one CTA) or 256
// (a CTA pair; `rank` selects the pair's lower or upper 128 rows).
__device__ __forceinline__ TileCoord tile_coord(int64_t i, const int* mt_prefix, int E, int n_tn,
                                                const int32_t* offsets_s, int BN,
                                                int rows_per_tile, int rank, int set) {
  // Find e with mt_prefix[e]*n_tn <= i < mt_prefix[e+1]*n_tn.
  int lo = 0, hi = E;  // invariant: prefix[lo]*n_tn <= i < prefix[hi]*n_tn
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (int64_t(mt_prefix[mid]) * n_tn <= i)
      lo = mid;
    else
      hi = mid;
  }
  const int e = lo;
  const int mts = mt_prefix[e + 1] - mt_prefix[e];
  const int64_t local = i - int64_t(mt_prefix[e]) * n_tn;
  const int nt = int(local / mts), mt = int(local % mts);
  TileCoord c;
  c.e = e;
  // A tail tile starts after the expert's whole 256-row tiles.
  const int tail0 = set == kTail ? ((offsets_s[e + 1] - offsets_s[e]) / 256) * 256 : 0;
  c.m0 = offsets_s[e] + tail0 + mt * rows_per_tile + rank * kTileM;
  c.m_end = offsets_s[e + 1] > offsets_s[e] ? offsets_s[e + 1] : offsets_s[e];
  c.n0 = nt * BN;
  return c;
}

template <int ACT>
__device__ __forceinline__ float epi_act(float u) {
  if constexpr (ACT == MOE_ACT_RELU) return u > 0.f ? u : 0.f;
  if constexpr (ACT == MOE_ACT_GELU_TANH)
    return 0.5f * u * (1.f + tc::tanh_fast(0.7978845608028654f * (u + 0.044715f * u * u * u)));
  return u;
}

// CK > 0: the second GEMM also runs the combine of [MoE 模型原理 §2.2, §5]
// in its epilogue (the combine folded into the expert GEMM, the other half of
// the fused permutation/dispatch kernel of [MoE Gate 分布式通信 mianshidashi,
// 06]).  A token's k expert rows are finished by different CTAs.  Before the
// GEMM, combine_prep_kernel sets every (token, column tile, column half)
// counter to the token's number of kept slots and writes y = 0 for tokens
// with none.  Each epilogue warp, once its rows of yd are stored and
// released, takes one count off per row; the warp whose decrement reaches
// zero sums the token's k rows of that column range in rank order in fp32
// (the arithmetic of combine_kernel, so y is identical bit for bit to the
// separate combine).  Nobody waits on anybody: the last arrival does the work.
// CK (2, 4, 8 or 16) bounds k, which sizes the per-token registers.
struct CombineArgs {
  const int32_t* slot_row;  // [T, k]
  const float* w;           // [T, k]
  __nv_bfloat16* y;         // [T, N]
  int* cnt;                 // [T, n_col_tiles, 2] arrivals still expected
  int k;
  int64_t T;
};

__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// The combine part of an epilogue warp of a combining GEMM, after the warp has stored rows
// row0 .. row0+31 of the tile, columns [c_lo, c_end) past n0: lane l arrives
// for row row0 + l; each lane whose arrival was the token's last loads the
// token's kept rows and weights (one round trip for all of them), then the
// warp sums two tokens at a time (16 lanes × 8 columns each).
template <int KMAX>
__device__ __forceinline__ void combine_rows(int m_end, int n0, int row0, int lane, int half,
                                             int c_lo, int c_end, int N, int BN, int64_t max_rows,
                                             const int32_t* __restrict__ row_token,
                                             const __nv_bfloat16* yd, const CombineArgs& cmb) {
  // Release: every lane fences its own stores of yd, then the warp meets, so
  // each row's stores (made by several lanes) are visible device-wide before
  // the lane that owns the row arrives.
  fence_acq_rel_gpu();
  __syncwarp();
  const int g = row0 + lane;
  int64_t t = -1;
  bool last = false;
  if (g < m_end) {
    const int32_t tt = row_token[g];
    if (tt >= 0 && int64_t(tt) < cmb.T) {
      t = tt;
      const int n_tn = (N + BN - 1) / BN;
      last = atomicAdd(cmb.cnt + (t * n_tn + n0 / BN) * 2 + half, -1) == 1;
    }
  }
  // Acquire: the completing decrement came after every other arrival's
  // release, so once the arriving lane has fenced and the warp has met, the
  // rows read below (from L2) are complete.
  fence_acq_rel_gpu();
  __syncwarp();
  unsigned m = __ballot_sync(0xffffffffu, last);
  if (!m) return;
  int32_t rows[KMAX];
  float wts[KMAX];
#pragma unroll
  for (int r = 0; r < KMAX; ++r) {
    rows[r] = -1;
    wts[r] = 0.f;
    if (last && r < cmb.k) {
      const int32_t sr = cmb.slot_row[t * cmb.k + r];
      if (sr >= 0 && int64_t(sr) < max_rows) {
        rows[r] = sr;
        wts[r] = cmb.w[t * cmb.k + r];
      }
    }
  }
  const int sub = lane & 15;
  const int col = c_lo + 8 * sub;
  const bool col_ok = col < c_end;
  while (m) {
    const int la = __ffs(m) - 1;
    m &= m - 1;
    int lb = la;
    bool two = false;
    if (m) {
      lb = __ffs(m) - 1;
      m &= m - 1;
      two = true;
    }
    const int src = lane < 16 ? la : lb;
    const int64_t tok = __shfl_sync(0xffffffffu, t, src);
    const bool active = (lane < 16 || two) && col_ok;
    float accv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) accv[i] = 0.f;
    // Ranks in groups of at most 8: all of a group's loads are issued before
    // any arithmetic; the sum still runs r = 0, 1, ... in order.
#pragma unroll
    for (int r0 = 0; r0 < KMAX; r0 += 8) {
      constexpr int G = KMAX < 8 ? KMAX : 8;
      int32_t rr[G];
      float ww[G];
      uint4 buf[G];
#pragma unroll
      for (int j = 0; j < G; ++j) {
        rr[j] = __shfl_sync(0xffffffffu, rows[r0 + j], src);
        ww[j] = __shfl_sync(0xffffffffu, wts[r0 + j], src);
        if (active && rr[j] >= 0)
          buf[j] = __ldcg(reinterpret_cast<const uint4*>(yd + int64_t(rr[j]) * N + n0 + col));
      }
#pragma unroll
      for (int j = 0; j < G; ++j) {
        float f[8];
        if (rr[j] >= 0) {
          const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&buf[j]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 p = __bfloat1622float2(hv[i]);
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) f[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) accv[i] = fmaf(ww[j], f[i], accv[i]);
      }
    }
    if (!active) continue;
    uint4 o;
    __nv_bfloat162* ho = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) ho[i] = __floats2bfloat162_rn(accv[2 * i], accv[2 * i + 1]);
    *reinterpret_cast<uint4*>(cmb.y + tok * N + n0 + col) = o;
  }
}

// Before a combining GEMM: cnt[t][nt][h] = kept slots of token t for every
// column tile nt and half h, and y[t] = 0 for a token with no kept slot.  One
// block per 256 tokens: each thread counts its token's kept slots, then the
// block writes its tokens' counters as one contiguous run.
__global__ void __launch_bounds__(256)
    combine_prep_kernel(int64_t T, int k, int per_token, int64_t max_rows, int64_t row_vecs,
                        const int32_t* __restrict__ slot_row, int* __restrict__ cnt,
                        uint4* __restrict__ y) {
  __shared__ int s_nk[256];
  pdl_wait();
  pdl_trigger();
  const int64_t t0 = int64_t(blockIdx.x) * 256;
  const int64_t t = t0 + threadIdx.x;
  int nk = 0;
  if (t < T)
    for (int r = 0; r < k; ++r) {
      const int32_t sr = slot_row[t * k + r];
      nk += (sr >= 0 && int64_t(sr) < max_rows) ? 1 : 0;
    }
  s_nk[threadIdx.x] = nk;
  __syncthreads();
  const int64_t n_tok = T - t0 < 256 ? T - t0 : 256;
  int* dst = cnt + t0 * per_token;
  for (int64_t i = threadIdx.x; i < n_tok * per_token; i += 256) dst[i] = s_nk[i / per_token];
  // y = 0 for the tokens of this block with no kept slot (a warp per token).
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = warp; j < n_tok; j += 8)
    if (s_nk[j] == 0)
      for (int64_t v = lane; v < row_vecs; v += 32) y[(t0 + j) * row_vecs + v] = make_uint4(0u, 0u, 0u, 0u);
}

// GATHER: the A rows are not read from a dispatch buffer but gathered from
// the token matrix x [gx_rows, K] through row_token (A[row] = x[row_token[row]],
// tmA a 64 × 1-box map over x): the permutation of [MoE 模型原理 §5] folded
// into the first GEMM's operand load, the fused permutation/dispatch kernel
// of [MoE Gate 分布式通信 mianshidashi, 06].  Every lane of warp 0 then
// issues TMA gather4 copies of four rows each, while lane 0 still loads B.
template <int ACT, bool PAIR, bool GATHER, int CK>
__global__ void __launch_bounds__(threads_for(GATHER), 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   int E, int N, int K, int BN, const int32_t* __restrict__ offsets,
                   const float* __restrict__ bias, __nv_bfloat16* __restrict__ out,
                   int64_t max_rows, int32_t* status, int stages, int set,
                   const int32_t* __restrict__ row_token, int64_t gx_rows, CombineArgs cmb) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
  __shared__ uint64_t tfull_bar[2], tempty_bar[2], drain_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_mt[kMaxExperts + 1];
  __shared__ int32_t s_off[kMaxExperts + 1];
  __shared__ int64_t s_tq[kTileQueue];
  __shared__ int s_tail_mt;  // the tail set's row tiles (pair launches)
  __shared__ uint64_t tq_full[kTileQueue], tq_empty[kTileQueue];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? tc::cluster_ctarank() : 0u;  // 0 = the pair's MMA issuer
  const int rows_per_tile = PAIR ? 2 * kTileM : kTileM;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int bn_cta = PAIR ? BN / 2 : BN;    // B rows staged by this CTA
  constexpr int KB = stage_kblocks(PAIR, GATHER);
  const uint32_t a_box = kTileM * kTileK * 2;             // one 64-wide k-block
  const uint32_t b_box = uint32_t(bn_cta) * kTileK * 2;
  const uint32_t a_bytes = KB * a_box;                     // one stage
  const uint32_t b_bytes = KB * b_box;
  uint8_t* sA = smem;                      // stages × a_bytes
  uint8_t* sB = smem + stages * a_bytes;   // stages × b_bytes
  uint8_t* sE = sB + stages * b_bytes;     // kEpiWarps × kEpiBufBytes

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      tc::mbar_init(&full_bar[s], 1);
      tc::mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&tfull_bar[a], 1);
      // One arrival per epilogue warp (of both CTAs of a pair).
      tc::mbar_init(&tempty_bar[a], PAIR ? 2 * kEpiWarps : kEpiWarps);
    }
    tc::mbar_init(&drain_bar, 1);
    for (int q = 0; q < kTileQueue; ++q) {
      tc::mbar_init(&tq_full[q], 1);
      tc::mbar_init(&tq_empty[q], 1 + kEpiWarps);  // the MMA warp and each epilogue warp
    }
    s_abort = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmA);
    tc::prefetch_tmap(&tmB);
  }
  // A pair allocates its tensor memory collectively (one warp in each CTA),
  // and the peer's barriers must be initialised before any copy or commit of
  // the pair can signal them: both need the peer CTA present.
  if constexpr (PAIR) tc::cluster_sync();
  if (warp == 1) {
    if constexpr (PAIR) {
      tc::tmem_alloc_pair(&s_tmem, kTmemCols);
      tc::tmem_relinquish_pair();
    } else {
      tc::tmem_alloc(&s_tmem, kTmemCols);
      tc::tmem_relinquish();
    }
  }
  // Launched with programmatic dependent launch: the A rows come from the
  // previous kernel, and the grid waits for it (griddepcontrol.wait) before
  // anything but the tile list.  offsets comes from a kernel before that one
  // (the dispatch, then the scatter or the first GEMM), and every kernel of
  // the layer waits for its own predecessor before it lets the next start,
  // so the tile list is built before the wait.  The gathering GEMM follows
  // the dispatch itself and waits first.  The tail launch starts while its
  // pair launch runs (which has waited already) and waits at its end.
  if (GATHER && set != kTail) {
    tc::grid_dependency_wait();
    tc::grid_launch_dependents();
  }
  // Per-expert m-tile prefix: warp 0 scans runs of experts, one run per lane.
  // Row offsets are clamped to [0, max_rows] so that no tile can reach
  // outside the buffers, whatever offsets holds; they are read through L2
  // (no stale L1 line from an earlier launch).
  if (warp == 0) {
    auto clamp_row = [&](int e) {
      const int32_t v = __ldcg(offsets + e);
      return int32_t(v < 0 ? 0 : (int64_t(v) > max_rows ? max_rows : v));
    };
    const int per = (E + 31) / 32;
    const int lo = lane * per, hi = min(E, lo + per);
    int run = 0, tail_run = 0;
    for (int e = lo; e < hi; ++e) {
      const int32_t a = clamp_row(e), b = clamp_row(e + 1);
      s_off[e] = a;
      run += tiles_in_set(b - a, set, rows_per_tile);
      if (set == kPairBody) tail_run += tiles_in_set(b - a, kTail, kTileM);
    }
    if (lane == 31) s_off[E] = clamp_row(E);
    tail_run = __reduce_add_sync(0xffffffffu, tail_run);
    if (lane == 0) s_tail_mt = tail_run;
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    int acc = incl - run;
    for (int e = lo; e < hi; ++e) {
      s_mt[e] = acc;
      const int32_t a = clamp_row(e), b = clamp_row(e + 1);
      acc += tiles_in_set(b - a, set, rows_per_tile);
    }
    if (lane == 31) s_mt[E] = incl;
  }
  if (!GATHER && set != kTail) {
    tc::grid_dependency_wait();
    tc::grid_launch_dependents();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = s_tmem;

  const int n_tn = (N + BN - 1) / BN;
  const int64_t total = int64_t(s_mt[E]) * n_tn;
  const int nk = (K + KB * kTileK - 1) / (KB * kTileK);  // stages per tile
  int64_t first_tile = PAIR ? blockIdx.x / 2 : blockIdx.x;
  int64_t tile_step = PAIR ? gridDim.x / 2 : gridDim.x;
  if (PAIR && !GATHER && set == kPairBody) {
    // When the tail launch that follows has work for kTailEarlySms SMs (two
    // tiles each), the last kTailEarlySms / 2 clusters take no tile and leave
    // at once, so the tail launch starts on their SMs beside this one.
    const int64_t clusters = gridDim.x / 2;
    if (int64_t(s_tail_mt) * n_tn >= 2 * kTailEarlySms && clusters > kTailEarlySms) {
      tile_step = clusters - kTailEarlySms / 2;
      if (first_tile >= tile_step) first_tile = total;
    }
  }
  volatile int* abort_flag = &s_abort;

  auto give_up = [&]() {
    *abort_flag = 1;
    set_status(status, MOE_ERR_TIMEOUT);
  };
  // Tile sequence of this CTA.  Static: first_tile, first_tile + tile_step,
  // ...  Dynamic (the one-CTA tail launch): the producer thread takes the
  // next tile from a counter in the workspace header and publishes it (or -1
  // when none is left) in a shared-memory queue that the MMA warp and the
  // epilogue warps read in the same order.
  const bool dyn = !PAIR && !GATHER && set == kTail;
  int* tail_ctr = reinterpret_cast<int*>(reinterpret_cast<char*>(status) + kWsTailTiles);
  auto static_tile = [&](int n) -> int64_t {
    const int64_t i = first_tile + int64_t(n) * tile_step;
    return i < total ? i : -1;
  };
  auto publish_tile = [&](int n) -> int64_t {  // producer thread
    if (!dyn) return static_tile(n);
    const int q = n % kTileQueue;
    if (!tc::mbar_wait(&tq_empty[q], uint32_t((n / kTileQueue) & 1) ^ 1u, abort_flag,
                       kWaitLimitNs)) {
      give_up();
      return -1;
    }
    const int64_t t = atomicAdd(tail_ctr, 1);
    const int64_t v = t < total ? t : -1;
    s_tq[q] = v;
    tc::mbar_arrive(&tq_full[q]);
    return v;
  };
  auto read_tile = [&](int n) -> int64_t {  // a whole consumer warp
    if (!dyn) return static_tile(n);
    const int q = n % kTileQueue;
    if (!__all_sync(0xffffffffu, tc::mbar_wait(&tq_full[q], uint32_t((n / kTileQueue) & 1),
                                                abort_flag, kWaitLimitNs))) {
      give_up();
      return -1;
    }
    const int64_t v = s_tq[q];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) tc::mbar_arrive(&tq_empty[q]);
    return v;
  };

  if (GATHER && (warp == 0 || warp >= kEpiWarp0 + kEpiWarps)) {
    // ---------------- gathering producer (whole warp) ----------------
    // Lane j gathers rows 4j .. 4j+3 of the 128-row A tile with one TMA
    // gather4 per k-block into bytes [512j, 512j + 512) of the stage: the
    // same 128-byte-swizzled layout a 64 × 128 box would write (each stage is
    // 1024-byte aligned).  Rows past the expert's end read token row 0 (they
    // are computed but never stored); lane 0 waits for the slot, posts the
    // stage's byte count and loads B.  Gathering warp gw (warp 0, then the
    // warps after the epilogue) serves the stages s with s mod kGatherWarps
    // == gw (all warps walk the same iteration sequence).
    const int gw = warp == 0 ? 0 : warp - (kEpiWarp0 + kEpiWarps) + 1;
    const int my_stage = gw / KB, my_half = gw % KB;
    const int nk64 = (K + kTileK - 1) / kTileK;  // 64-wide k-blocks
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int64_t i = first_tile; i < total && ok; i += tile_step) {
      const TileCoord c =
          tile_coord(i, s_mt, E, n_tn, s_off, BN, rows_per_tile, int(rank), set);
      int32_t t4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int g = c.m0 + 4 * lane + q;
        const int32_t t = g < c.m_end ? row_token[g] : 0;
        t4[q] = (t >= 0 && int64_t(t) < gx_rows) ? t : 0;
      }
      for (int kb = 0; kb < nk; ++kb) {
        if (stage != my_stage) {  // another warp's stage
          ++issued;
          if (++stage == stages) stage = 0, phase ^= 1u;
          continue;
        }
        int free_slot = 1;
        if (lane == 0)
          free_slot = tc::mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, kWaitLimitNs);
        if (!__shfl_sync(0xffffffffu, free_slot, 0)) {
          if (lane == 0) give_up();
          ok = false;
          break;
        }
        // This warp's k-block of the stage; a half past K (K/64 odd) is
        // neither copied nor multiplied, and the stage's byte count (posted
        // by the half-0 warp) leaves it out.
        const int kblk = kb * KB + my_half;
        const int halves = min(KB, nk64 - kb * KB);
        const uint32_t stage_tx = uint32_t(halves) * (a_box + b_box);
        uint8_t* dst = sA + stage * a_bytes + my_half * a_box + lane * 512;
        uint8_t* dstB = sB + stage * b_bytes + my_half * b_box;
        if constexpr (PAIR) {
          const uint32_t bar = tc::mapa(tc::smem_u32(&full_bar[stage]), 0);
          if (lane == 0) {
            if (rank == 0 && my_half == 0) tc::mbar_arrive_expect_tx(&full_bar[stage], 2 * stage_tx);
            if (kblk < nk64)
              tc::tma_load_3d_pair(&tmB, bar, dstB, kblk * kTileK, c.n0 + int(rank) * bn_cta,
                                   c.e);
          }
          __syncwarp();
          if (kblk < nk64)
            tc::tma_gather4_pair(&tmA, bar, dst, kblk * kTileK, t4[0], t4[1], t4[2], t4[3]);
        } else {
          if (lane == 0) {
            if (my_half == 0) tc::mbar_arrive_expect_tx(&full_bar[stage], stage_tx);
            if (kblk < nk64)
              tc::tma_load_3d(&tmB, &full_bar[stage], dstB, kblk * kTileK, c.n0, c.e);
          }
          __syncwarp();
          if (kblk < nk64)
            tc::tma_gather4(&tmA, &full_bar[stage], dst, kblk * kTileK, t4[0], t4[1], t4[2],
                            t4[3]);
        }
        ++issued;
        if (++stage == stages) stage = 0, phase ^= 1u;
      }
    }
    // Drain as the TMA producer does: the last `stages` stages (of every
    // gathering warp) land before the CTA exits.
    if (gw == 0 && rank == 0 && lane == 0) {
      const int64_t first = issued > stages ? issued - stages : 0;
      for (int64_t j = first; j < issued; ++j)
        tc::mbar_wait(&full_bar[j % stages], uint32_t((j / stages) & 1), nullptr, kWaitLimitNs);
    }
  } else if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool ok = true;
    int n_tile = 0;
    for (int64_t i = publish_tile(0); i >= 0 && ok; i = publish_tile(++n_tile)) {
      const TileCoord c =
          tile_coord(i, s_mt, E, n_tn, s_off, BN, rows_per_tile, int(rank), set);
      for (int kb = 0; kb < nk; ++kb) {
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
          // A k-block past K (K/64 odd) arrives as zeros, which add nothing.
#pragma unroll
          for (int h = 0; h < KB; ++h) {
            const int kx = (kb * KB + h) * kTileK;
            tc::tma_load_2d_pair(&tmA, bar, sA + stage * a_bytes + h * a_box, kx, c.m0);
            tc::tma_load_3d_pair(&tmB, bar, sB + stage * b_bytes + h * b_box, kx,
                                 c.n0 + int(rank) * bn_cta, c.e);
          }
        } else {
          tc::mbar_arrive_expect_tx(&full_bar[stage], a_bytes + b_bytes);
#pragma unroll
          for (int h = 0; h < KB; ++h) {
            const int kx = (kb * KB + h) * kTileK;
            tc::tma_load_2d(&tmA, &full_bar[stage], sA + stage * a_bytes + h * a_box, kx, c.m0);
            tc::tma_load_3d(&tmB, &full_bar[stage], sB + stage * b_bytes + h * b_box, kx, c.n0,
                            c.e);
          }
        }
        ++issued;
        if (++stage == stages) stage = 0, phase ^= 1u;
      }
    }
    // Drain: the last `stages` copies must land before the CTA exits (on the
    // normal path the MMA issuer has consumed them all).  In a pair the even
    // CTA's full barriers track the copies of both CTAs.
    if (rank == 0) {
      const int64_t first = issued > stages ? issued - stages : 0;
      for (int64_t j = first; j < issued; ++j)
        tc::mbar_wait(&full_bar[j % stages], uint32_t((j / stages) & 1), nullptr, kWaitLimitNs);
    }
  } else if (warp == 1 && rank == 0) {
    // ---------------- MMA issuer (whole warp, one elected lane issues) -----
    const uint32_t idesc = tc::idesc_bf16_f32(rows_per_tile, BN);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    int n_tile = 0;
    for (int64_t i = read_tile(0); i >= 0 && ok; i = read_tile(++n_tile)) {
      // Waits are taken by every lane and agreed on, so the warp stays
      // converged and its operands warp-uniform.
      const bool free_acc = __all_sync(
          0xffffffffu, PAIR ? tc::mbar_wait_cluster(&tempty_bar[acc], acc_phase ^ 1u, abort_flag,
                                                    kWaitLimitNs)
                            : tc::mbar_wait(&tempty_bar[acc], acc_phase ^ 1u, abort_flag,
                                            kWaitLimitNs));
      if (!free_acc) {
        give_up();
        break;
      }
      tc::fence_after_sync();
      const uint32_t d_tmem = tmem_base + uint32_t(acc * kAccCols);
      for (int kb = 0; kb < nk; ++kb) {
        if (!__all_sync(0xffffffffu,
                        tc::mbar_wait(&full_bar[stage], phase, abort_flag, kWaitLimitNs))) {
          give_up();
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t a0 = tc::smem_u32(sA + stage * a_bytes);
        const uint32_t b0 = tc::smem_u32(sB + stage * b_bytes);
        const uint64_t ad0 = tc::sdesc_kmajor_sw128(a0), bd0 = tc::sdesc_kmajor_sw128(b0);
        // The gathering producer copies no k-block past K (K/64 odd).
        const int mma_steps =
            GATHER ? min(KB, (K + kTileK - 1) / kTileK - kb * KB) * (kTileK / 16) : KB * kTileK / 16;
#pragma unroll
        for (int j = 0; j < KB * kTileK / 16; ++j) {
          if (GATHER && j >= mma_steps) break;
          const uint32_t h = uint32_t(j / (kTileK / 16)), q = uint32_t(j % (kTileK / 16));
          const uint64_t ad = tc::sdesc_advance(ad0, h * a_box + q * 32);
          const uint64_t bd = tc::sdesc_advance(bd0, h * b_box + q * 32);
          if constexpr (PAIR)
            tc::mma_bf16_pair_w(d_tmem, ad, bd, idesc, (kb | j) != 0);
          else
            tc::mma_bf16_w(d_tmem, ad, bd, idesc, (kb | j) != 0);
        }
        if constexpr (PAIR)
          tc::mma_commit_pair_mc_w(&empty_bar[stage], 0x3);
        else
          tc::mma_commit_w(&empty_bar[stage]);
        if (++stage == stages) stage = 0, phase ^= 1u;
      }
      if (!ok) break;
      if constexpr (PAIR)
        tc::mma_commit_pair_mc_w(&tfull_bar[acc], 0x3);
      else
        tc::mma_commit_w(&tfull_bar[acc]);
      if (++acc == 2) acc = 0, acc_phase ^= 1u;
    }
    // Drain: wait until every MMA this warp issued has completed.
    if constexpr (PAIR)
      tc::mma_commit_pair_w(&drain_bar);
    else
      tc::mma_commit_w(&drain_bar);
    tc::mbar_wait(&drain_bar, 0, nullptr, kWaitLimitNs);
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps) {
    // ---------------- epilogue ----------------
    const int quarter = warp & 3;              // TMEM lanes [32·quarter, 32·quarter+32)
    const int half = (warp - kEpiWarp0) >> 2;  // columns [c_lo, c_hi) of the tile
    const int hb = ((BN / 2 + 15) / 16) * 16;
    const int c_lo = half * hb, c_hi = min(BN, c_lo + hb);
    uint8_t* buf = sE + (warp - kEpiWarp0) * kEpiBufBytes;
    const uint32_t buf_s = tc::smem_u32(buf);
    int acc = 0;
    uint32_t acc_phase = 0;
    int n_tile = 0;
    for (int64_t i = read_tile(0); i >= 0; i = read_tile(++n_tile)) {
      const TileCoord c =
          tile_coord(i, s_mt, E, n_tn, s_off, BN, rows_per_tile, int(rank), set);
      // The tensor-memory loads below are warp-collective: the whole warp
      // takes the same branch.
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&tfull_bar[acc], acc_phase, abort_flag,
                                                 kWaitLimitNs))) {
        give_up();
        break;
      }
      tc::fence_after_sync();
      const int ncols = min(BN, N - c.n0);
      const float* bias_e = bias + int64_t(c.e) * N + c.n0;
      const int row0 = c.m0 + quarter * 32;
      const uint32_t t_row = tmem_base + (uint32_t(quarter * 32) << 16) + uint32_t(acc * kAccCols);
      for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
        uint32_t r[32];
        tc::tmem_ld_x32(t_row + uint32_t(c0), r);
        float b[32];
        if (c0 + 32 <= ncols) {
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 q = __ldg(reinterpret_cast<const float4*>(bias_e + c0 + j));
            b[j] = q.x, b[j + 1] = q.y, b[j + 2] = q.z, b[j + 3] = q.w;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) b[j] = c0 + j < ncols ? __ldg(bias_e + c0 + j) : 0.f;
        }
        tc::tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float u0 = epi_act<ACT>(__uint_as_float(r[2 * j]) + b[2 * j]);
          const float u1 = epi_act<ACT>(__uint_as_float(r[2 * j + 1]) + b[2 * j + 1]);
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(u0, u1);
          pk[j] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        // Row `lane` of the warp's 32×32 block -> shared buffer (64 bytes per
        // row, 16-byte pieces XOR-swizzled by row so that each group of 8
        // lanes hits distinct banks).
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t addr = buf_s + uint32_t(lane * 64 + ((q ^ ((lane >> 1) & 3)) * 16));
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * q]),
                       "r"(pk[4 * q + 1]), "r"(pk[4 * q + 2]), "r"(pk[4 * q + 3])
                       : "memory");
        }
        __syncwarp();
        // Read back 8 rows × 4 pieces per step: each store covers 8 rows of
        // 64 contiguous bytes.
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int rr = it * 8 + (lane >> 2), q = lane & 3;
          const uint32_t addr = buf_s + uint32_t(rr * 64 + ((q ^ ((rr >> 1) & 3)) * 16));
          uint4 v;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                       : "r"(addr)
                       : "memory");
          const int grow = row0 + rr, gcol = c0 + q * 8;
          if (grow < c.m_end && gcol < ncols)
            *reinterpret_cast<uint4*>(out + int64_t(grow) * N + c.n0 + gcol) = v;
        }
        __syncwarp();
      }
      // This warp is done reading the accumulator: one arrival per warp on
      // the MMA issuer's barrier (in the even CTA of a pair).
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if constexpr (PAIR)
          tc::mbar_arrive_cluster(tc::mapa(tc::smem_u32(&tempty_bar[acc]), 0));
        else
          tc::mbar_arrive(&tempty_bar[acc]);
      }
      if (++acc == 2) acc = 0, acc_phase ^= 1u;
      if constexpr (CK > 0) {
        const int c_end = min(c_hi, ncols);
        if (c_lo < c_end)
          combine_rows<CK>(c.m_end, c.n0, row0, lane, half, c_lo, c_end, N, BN, max_rows,
                           row_token, out, cmb);
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
      tc::tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tc::tmem_dealloc(tmem_base, kTmemCols);
  }
  // The last CTA of a dynamic tail launch to finish clears the tile counter
  // for the next launch (every CTA has taken its last tile by now).
  if (dyn && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(tail_ctr + 1, 1) == int(gridDim.x) - 1) {
      atomicExch(tail_ctr, 0);
      atomicExch(tail_ctr + 1, 0);
    }
  }
  // A tail launch that started early does not finish before the pair launch
  // it overlapped: work after it in the stream sees every tile.
  if (set == kTail) tc::grid_dependency_wait();
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

// Column-tile width: as many tiles as 256-wide ones would need, each the
// narrowest multiple of 16 that still covers N (N = 1408: six tiles of 240
// columns instead of six of 256 with half of the last one masked).  Fewer,
// narrower tiles keep each SM's A stream feeding as many output columns as
// possible: eight exact tiles of 176 columns measured 11% slower than six of
// 256 at N = 1408.
int pick_bn(int N) {
  if (N <= 256) return ((N + 15) / 16) * 16;
  const int tiles = (N + 255) / 256;
  return ((N + tiles - 1) / tiles + 15) / 16 * 16;
}

// The 2-SM variant is the default; MOE_GEMM_PAIR=0 selects the 1-SM kernel
// (a cross-check in tests).
bool use_pair() {
  const char* v = std::getenv("MOE_GEMM_PAIR");
  return !(v && std::strcmp(v, "0") == 0);
}

// Gathered A rows (GATHER): row_token and the rows of the token matrix,
// else unused.
struct Gather {
  const int32_t* row_token;
  int64_t gx_rows;
};

template <bool PAIR, bool GATHER, bool COMBINE>
cudaError_t launch_variant(int act, const CUtensorMap& tmA, const CUtensorMap& tmB, int E, int N,
                           int K, int BN, const int32_t* offsets, const float* bias, void* out,
                           int64_t max_rows, int32_t* status, int set, const Gather& g,
                           const CombineArgs& cmb, cudaStream_t st) {
  const int sms = device_sms();
  const size_t static_smem = kernel_static_smem(
      reinterpret_cast<const void*>(gemm_tc_kernel<kActNone, PAIR, false, 0>));
  // As many pipeline stages as fit beside the epilogue buffers and the
  // kernel's static shared memory.
  const int bn_cta = PAIR ? BN / 2 : BN;
  const size_t stage_bytes =
      size_t(stage_kblocks(PAIR, GATHER)) * (size_t(kTileM) + bn_cta) * kTileK * 2;
  const size_t fixed = 1024 + size_t(kEpiWarps) * kEpiBufBytes;
  const size_t budget = size_t(device_smem_optin()) - static_smem;
  int stages = budget > fixed ? int((budget - fixed) / stage_bytes) : 0;
  if (stages > kMaxStages) stages = kMaxStages;
  // Every stage half needs its own gathering warp.
  if (GATHER && stages * stage_kblocks(PAIR, true) > kGatherWarps)
    stages = kGatherWarps / stage_kblocks(PAIR, true);
  if (stages < 2) return cudaErrorInvalidValue;
  const size_t smem = fixed + size_t(stages) * stage_bytes;
  auto run = [&](auto kernel) {
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kernel), smem);
    if (e != cudaSuccess) return e;
    unsigned grid = unsigned(sms);
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(threads_for(GATHER));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    if constexpr (PAIR) {
      // Persistent grid: as many CTA pairs as can be resident at once.
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      cfg.gridDim = dim3(2);
      int clusters = 0;
      e = max_active_clusters(reinterpret_cast<const void*>(kernel), cfg, &clusters);
      if (e != cudaSuccess) return e;
      if (clusters < 1) return cudaErrorInvalidConfiguration;
      grid = unsigned(2 * clusters);
    }
    cfg.gridDim = dim3(grid);
    // Programmatic dependent launch on every launch (see the kernel's
    // prologue): the grid is scheduled while the previous kernel finishes.
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs += 1;
    e = cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, E, N, K, BN, offsets, bias,
                           static_cast<__nv_bfloat16*>(out), max_rows, status, stages, set,
                           g.row_token, g.gx_rows, cmb);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  };
  if constexpr (GATHER) {
    // Only the first GEMM gathers, and it always has an activation.
    return act == MOE_ACT_RELU        ? run(gemm_tc_kernel<MOE_ACT_RELU, PAIR, true, 0>)
           : act == MOE_ACT_GELU_TANH ? run(gemm_tc_kernel<MOE_ACT_GELU_TANH, PAIR, true, 0>)
                                      : cudaErrorInvalidValue;
  } else if constexpr (COMBINE) {
    // Only the second GEMM combines, and it has no activation; the combine
    // holds up to 2, 4, 8 or 16 ranks per token.
    if (act >= 0) return cudaErrorInvalidValue;
    return cmb.k <= 2   ? run(gemm_tc_kernel<kActNone, PAIR, false, 2>)
           : cmb.k <= 4 ? run(gemm_tc_kernel<kActNone, PAIR, false, 4>)
           : cmb.k <= 8 ? run(gemm_tc_kernel<kActNone, PAIR, false, 8>)
                        : run(gemm_tc_kernel<kActNone, PAIR, false, 16>);
  } else {
    return act == MOE_ACT_RELU        ? run(gemm_tc_kernel<MOE_ACT_RELU, PAIR, false, 0>)
           : act == MOE_ACT_GELU_TANH ? run(gemm_tc_kernel<MOE_ACT_GELU_TANH, PAIR, false, 0>)
                                      : run(gemm_tc_kernel<kActNone, PAIR, false, 0>);
  }
}

template <bool GATHER, bool COMBINE>
cudaError_t launch_sets(int act, const CUtensorMap& tmA, const CUtensorMap& tmB_cta,
                        const CUtensorMap* tmB_pair, int E, int N, int K, int BN,
                        const int32_t* offsets, const float* bias, void* out, int64_t max_rows,
                        int32_t* status, const Gather& g, const CombineArgs& cmb,
                        cudaStream_t st) {
  cudaError_t err;
  if (tmB_pair && E >= kTailSplitMinExperts) {
    // CTA pairs take every expert's whole 256-row tiles (and a last one with
    // more than 128 rows); one-CTA tiles take the remaining 1..128 rows, so
    // no pair computes a 128-row half that lies past its expert's end.
    err = launch_variant<true, GATHER, COMBINE>(act, tmA, *tmB_pair, E, N, K, BN, offsets, bias,
                                                out, max_rows, status, kPairBody, g, cmb, st);
    if (err != cudaSuccess) return err;
    count_launch();
    err = launch_variant<false, GATHER, COMBINE>(act, tmA, tmB_cta, E, N, K, BN, offsets, bias,
                                                 out, max_rows, status, kTail, g, cmb, st);
  } else if (tmB_pair) {
    err = launch_variant<true, GATHER, COMBINE>(act, tmA, *tmB_pair, E, N, K, BN, offsets, bias,
                                                out, max_rows, status, kAllTiles, g, cmb, st);
  } else {
    err = launch_variant<false, GATHER, COMBINE>(act, tmA, tmB_cta, E, N, K, BN, offsets, bias,
                                                 out, max_rows, status, kAllTiles, g, cmb, st);
  }
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaSuccess;
}

}  // namespace

namespace {

// A tensor map over A [rows, K] (K contiguous): 64 × 128 boxes over the
// dispatch buffer, or 64 × 1 boxes (the gather4 form) over the token matrix.
bool encode_a(EncodeTiledFn encode, CUtensorMap* m, const void* A, int K, int64_t rows,
              int box_rows) {
  const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(K) * 2};
  const cuuint32_t box[2] = {kTileK, cuuint32_t(box_rows)};
  const cuuint32_t es[2] = {1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(A), dims, strides, box,
                es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// B tiles of BN rows (one CTA) or BN/2 rows (each CTA of a pair).
bool encode_b(EncodeTiledFn encode, CUtensorMap* m, const void* B, int E, int N, int K,
              int box_rows) {
  const cuuint64_t dims[3] = {cuuint64_t(K), cuuint64_t(N), cuuint64_t(E)};
  const cuuint64_t strides[2] = {cuuint64_t(K) * 2, cuuint64_t(N) * K * 2};
  const cuuint32_t box[3] = {kTileK, cuuint32_t(box_rows), 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(B), dims, strides, box,
                es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool GATHER, bool COMBINE>
cudaError_t launch_gemm(int E, int N, int K, int64_t max_rows, const int32_t* offsets,
                        const void* A, int64_t a_rows, const void* B, const float* bias, int act,
                        void* out, int32_t* status, const Gather& g, const CombineArgs& cmb,
                        cudaStream_t st) {
  if (E > kMaxExperts) return cudaErrorInvalidValue;
  EncodeTiledFn encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  const int BN = pick_bn(N);
  CUtensorMap tmA, tmB_cta, tmB_pair;
  if (!encode_a(encode, &tmA, A, K, a_rows, GATHER ? 1 : kTileM)) return cudaErrorInvalidValue;
  if (!encode_b(encode, &tmB_cta, B, E, N, K, BN)) return cudaErrorInvalidValue;
  const bool pair = use_pair();
  if (pair && !encode_b(encode, &tmB_pair, B, E, N, K, BN / 2)) return cudaErrorInvalidValue;
  return launch_sets<GATHER, COMBINE>(act, tmA, tmB_cta, pair ? &tmB_pair : nullptr, E, N, K, BN,
                                      offsets, bias, out, max_rows, status, g, cmb, st);
}

}  // namespace

cudaError_t launch_gemm_tc(int E, int N, int K, int64_t max_rows, const int32_t* offsets,
                           const void* A, const void* B, const float* bias, int act, void* out,
                           int32_t* status, cudaStream_t st) {
  const Gather none{nullptr, 0};
  const CombineArgs no_cmb{nullptr, nullptr, nullptr, nullptr, 0, 0};
  return launch_gemm<false, false>(E, N, K, max_rows, offsets, A, max_rows, B, bias, act, out,
                                   status, none, no_cmb, st);
}

cudaError_t launch_gemm_tc_gather(int E, int N, int K, int64_t max_rows, const int32_t* offsets,
                                  const void* x, int64_t T, const int32_t* row_token,
                                  const void* B, const float* bias, int act, void* out,
                                  int32_t* status, cudaStream_t st) {
  if (act != MOE_ACT_RELU && act != MOE_ACT_GELU_TANH) return cudaErrorInvalidValue;
  const Gather g{row_token, T};
  const CombineArgs no_cmb{nullptr, nullptr, nullptr, nullptr, 0, 0};
  return launch_gemm<true, false>(E, N, K, max_rows, offsets, x, T, B, bias, act, out, status, g,
                                  no_cmb, st);
}

int gemm_tc_bn(int N) { return pick_bn(N); }

cudaError_t launch_gemm_tc_combine(int E, int N, int K, int64_t max_rows, const int32_t* offsets,
                                   const void* A, const void* B, const float* bias, void* yd,
                                   int64_t T, int k, const int32_t* row_token,
                                   const int32_t* slot_row, const float* w, void* y, int* cnt,
                                   int32_t* status, cudaStream_t st) {
  if (N % 8 != 0) return cudaErrorInvalidValue;
  const int BN = pick_bn(N);
  const int per_token = 2 * ((N + BN - 1) / BN);
  cudaError_t e = launch_pdl(combine_prep_kernel, dim3(unsigned((T + 255) / 256)), dim3(256), 0,
                             st, T, k, per_token, max_rows, int64_t(N / 8), slot_row, cnt,
                             static_cast<uint4*>(y));
  count_launch();
  if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) return e;
  const Gather g{row_token, 0};
  const CombineArgs cmb{slot_row, w, static_cast<__nv_bfloat16*>(y), cnt, k, T};
  return launch_gemm<false, true>(E, N, K, max_rows, offsets, A, max_rows, B, bias, -1, yd,
                                  status, g, cmb, st);
}

}  // namespace moe
