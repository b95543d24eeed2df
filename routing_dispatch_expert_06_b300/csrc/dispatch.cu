// Dispatch: expert histogram, capacity, first-come positions and the token
// permutation into the per-expert buffer.
//
// [MoE 模型原理 §4.1] C = ceil(c·T·k/E).
// [MoE 模型原理 §4.2] each expert keeps at most C slots, the earliest ones;
//   capacity is per expert and never moves to another expert.
// [MoE 模型原理 §4.3] overflow slots are dropped (the residual path).
// [MoE 模型原理 §5]   kept slots are gathered into one contiguous buffer,
//   expert by expert ("dispatch_mask or an equivalent index").
//
// Position of slot (t, r) routed to expert e = number of earlier tokens t' < t
// that also routed to e (a token selects each expert at most once, so the
// (token, rank) order within an expert is plain token order).  It is built in
// integer passes and never materialises a T×E one-hot mask:
//   1. histogram per chunk of 256 tokens         chunk_counts[chunk][e]
//   2. per-expert exclusive scan over chunks     chunk_counts -> chunk bases,
//      counts[e], kept[e] = min(counts[e], C) — done by the last histogram
//      block to finish when a completion counter is given, else by a
//      separate kernel
//   3. per chunk: expert offsets (scan of kept), per-warp bases, then each
//      warp walks the slots of its 32 tokens in (token, rank) order, 32 slots
//      per step: slot_row, row_token
// and a fourth, bandwidth-bound pass copies each token row once from x and
// writes it to every kept slot with 16-byte vectors.
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kDispatchThreads = 256;  // 8 warps × 32 tokens = one chunk
static_assert(kDispatchThreads == kChunkTokens, "one token per thread in a chunk");
static_assert(kDispatchThreads == kAuxThreads, "the last histogram block runs the statistics");

// Per-expert exclusive scan over the chunk histograms (in place), the total
// count and kept = min(count, C), by one block; with cap_base (a second fill
// round into the room C - cap_base[e] left by the first), kept =
// cap_base[e] + min(count, C - cap_base[e]).  A group of tpe lanes (a power
// of two, as many as the block holds for E experts, at most 32) scans one
// expert; each lane loads U consecutive chunk counts at once (U = 8, or 32
// when a group has fewer than 4 lanes, i.e. many experts), so an expert's
// n_chunks take ceil(n_chunks / (U·tpe)) rounds of overlapping loads.
template <int U>
__device__ void scan_chunks_rounds(int64_t n_chunks, int E, int64_t C, int tpe,
                                   int32_t* __restrict__ chunk_counts,
                                   int32_t* __restrict__ counts, int32_t* __restrict__ kept,
                                   const int32_t* __restrict__ cap_base) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & (tpe - 1);
  const int group = threadIdx.x / tpe;
  const int ngroups = blockDim.x / tpe;
  const unsigned gmask =
      tpe == 32 ? 0xffffffffu : (((1u << tpe) - 1u) << (lane & ~(tpe - 1)));
  for (int e = group; e < E; e += ngroups) {
    int32_t carry = 0;
    for (int64_t base = 0; base < n_chunks; base += int64_t(tpe) * U) {
      const int64_t c0 = base + int64_t(sub) * U;
      int32_t v[U];
      int32_t tot = 0;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        v[u] = c0 + u < n_chunks ? __ldcg(chunk_counts + (c0 + u) * E + e) : 0;
        tot += v[u];
      }
      int32_t incl = tot;
      for (int o = 1; o < tpe; o <<= 1) {
        const int32_t up = __shfl_up_sync(gmask, incl, o, tpe);
        if (sub >= o) incl += up;
      }
      int32_t run = carry + incl - tot;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (c0 + u < n_chunks) chunk_counts[(c0 + u) * E + e] = run;
        run += v[u];
      }
      carry += __shfl_sync(gmask, incl, tpe - 1, tpe);
    }
    if (sub == 0) {
      counts[e] = carry;
      const int32_t base = cap_base ? cap_base[e] : 0;
      const int64_t room = C - base;
      kept[e] = base + int32_t(carry < room ? carry : room);
    }
  }
}

__device__ void scan_chunks_by_expert(int64_t n_chunks, int E, int64_t C,
                                      int32_t* __restrict__ chunk_counts,
                                      int32_t* __restrict__ counts, int32_t* __restrict__ kept,
                                      const int32_t* __restrict__ cap_base) {
  int tpe = 32;
  while (tpe > 1 && tpe * E > int(blockDim.x)) tpe >>= 1;
  if (tpe >= 4)
    scan_chunks_rounds<8>(n_chunks, E, C, tpe, chunk_counts, counts, kept, cap_base);
  else
    scan_chunks_rounds<32>(n_chunks, E, C, tpe, chunk_counts, counts, kept, cap_base);
}

// Histogram of one chunk; with a completion counter, the last block to
// finish also runs the per-expert scan.  skip_neg: ids < 0 are not counted
// (the second round of a reroute); cap_base: see scan_chunks_by_expert.
__device__ __forceinline__ void histogram_body(int64_t T, int E, int k,
                                               const int32_t* __restrict__ ids,
                                               int32_t* __restrict__ chunk_counts,
                                               int32_t* status, int* counter, int64_t C,
                                               int32_t* __restrict__ counts,
                                               int32_t* __restrict__ kept, const AuxArgs& aux,
                                               int skip_neg, const int32_t* __restrict__ cap_base,
                                               int32_t* hist) {
  __shared__ int s_last;
  __shared__ float s_red[kAuxThreads];
  __shared__ unsigned long long s_kept_sum;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t t = int64_t(blockIdx.x) * kChunkTokens + threadIdx.x;
  if (t < T) {
    for (int r = 0; r < k; ++r) {
      const int e = ids[t * k + r];
      if (e >= 0 && e < E)
        atomicAdd(&hist[e], 1);
      else if (!(skip_neg && e < 0))
        set_status(status, MOE_ERR_INVALID_ARG);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_counts[int64_t(blockIdx.x) * E + e] = hist[e];
  if (counter && last_block_to_finish(counter, &s_last)) {
    scan_chunks_by_expert(gridDim.x, E, C, chunk_counts, counts, kept, cap_base);
    const int32_t* counts_f = aux.counts_f ? aux.counts_f : counts;
    if (aux.f) {
      if (aux.psum_fixed) psum_from_fixed(E, aux.psum_fixed, aux.psum);
      __syncthreads();
      aux_stats_block(E, T, aux.alpha, counts_f, aux.psum, aux.f, aux.pbar, aux.l_aux, s_red);
    }
    if (aux.health) {
      __syncthreads();
      routing_health_block(E, T, k, counts_f, kept, aux.health, s_red, &s_kept_sum);
    }
  }
}

__global__ void __launch_bounds__(kDispatchThreads)
    histogram_kernel(int64_t T, int E, int k, const int32_t* __restrict__ ids,
                     int32_t* __restrict__ chunk_counts, int32_t* status, int* counter,
                     int64_t C, int32_t* __restrict__ counts, int32_t* __restrict__ kept,
                     AuxArgs aux, int skip_neg, const int32_t* __restrict__ cap_base) {
  extern __shared__ int32_t hist[];
  pdl_wait();
  pdl_trigger();
  histogram_body(T, E, k, ids, chunk_counts, status, counter, C, counts, kept, aux, skip_neg,
                 cap_base, hist);
}

// One CTA per expert: exclusive scan of that expert's chunk counts (in place),
// total count and kept = min(count, C).
__global__ void __launch_bounds__(256)
    expert_scan_kernel(int64_t n_chunks, int E, int64_t C, int32_t* __restrict__ chunk_counts,
                       int32_t* __restrict__ counts, int32_t* __restrict__ kept) {
  __shared__ int32_t warp_tot[8];
  __shared__ int32_t carry;
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int64_t base = 0; base < n_chunks; base += blockDim.x) {
    const int64_t ch = base + threadIdx.x;
    const int32_t v = ch < n_chunks ? chunk_counts[ch * E + e] : 0;
    int32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int32_t before = carry;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    if (ch < n_chunks) chunk_counts[ch * E + e] = before + incl - v;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = before + incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    counts[e] = carry;
    kept[e] = int32_t(carry < C ? carry : C);
  }
}

// One CTA per chunk of 256 tokens; warp w owns tokens [32w, 32w+32) of it.
// Dynamic shared memory: off[E+1] | wbase[8][E] | the chunk's ids [256·k].
// off[e] = Σ_{e' < e} v[e'] for e <= E (off[E] = total), by one block of
// kDispatchThreads threads: thread i sums a run of consecutive entries, then a
// block scan (warp shuffles, then the 8 warp totals) gives each run's start.
// Ends with the block synchronised.
__device__ __forceinline__ void block_exclusive_scan(int E, const int32_t* __restrict__ v,
                                                     int32_t* off, int32_t* part) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (E + kDispatchThreads - 1) / kDispatchThreads;
  const int lo = tid * per, hi = min(E, lo + per);
  int32_t run = 0;
  for (int e = lo; e < hi; ++e) run += v[e];
  int32_t incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) part[warp] = incl;
  __syncthreads();
  int32_t before = 0;
  for (int w = 0; w < warp; ++w) before += part[w];
  if (tid == kDispatchThreads - 1) off[E] = before + incl;
  int32_t acc = before + incl - run;
  for (int e = lo; e < hi; ++e) {
    off[e] = acc;
    acc += v[e];
  }
  __syncthreads();
}

// Walk warp w's slots of the chunk starting at token chunk0 in (token, rank)
// order, 32 at a time: warp w owns the slots of its 32 tokens, s = t·k + r,
// so step i takes slots 32·w·k + 32·i + lane (k steps).  A slot's position is
// its expert's count so far (my[e], the warp's base on entry) plus the number
// of earlier lanes of the step with the same expert (match.any groups; this
// also covers a token naming one expert at two ranks), and the group's first
// lane advances my[e] by the group size.  off: expert offsets (positions_only:
// the per-expert capacity).
__device__ __forceinline__ void walk_slots(int64_t T, int E, int k, int64_t C, int64_t chunk0,
                                           const int32_t* s_ids, int32_t* my, const int32_t* off,
                                           int32_t* __restrict__ slot_row,
                                           int32_t* __restrict__ row_token, int positions_only) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t chunk_slots = (T - chunk0 < kChunkTokens ? T - chunk0 : kChunkTokens) * k;
  for (int it = 0; it < k; ++it) {
    const int64_t ls = int64_t(warp) * 32 * k + int64_t(it) * 32 + lane;  // slot within chunk
    const bool in = ls < chunk_slots;
    const int e = in ? s_ids[ls] : -1;
    const bool valid = e >= 0 && e < E;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : E + lane);
    const int32_t before = __popc(peers & ((1u << lane) - 1u));
    const int32_t base = valid ? my[e] : 0;
    __syncwarp();
    if (valid && before == 0) my[e] = base + __popc(peers);
    __syncwarp();
    if (in) {
      const int64_t s_glob = chunk0 * k + ls;
      int32_t row = -1;
      if (valid) {
        const int32_t pos = base + before;
        if (positions_only) {
          row = pos < off[e] ? pos : -1;  // off[e] holds the capacity here
        } else if (pos < C) {
          row = off[e] + pos;
          row_token[row] = int32_t(s_glob / k);
        }
      }
      slot_row[s_glob] = row;
    }
  }
}

__device__ __forceinline__ void assign_body(int64_t T, int E, int k, int64_t C,
                                            const int32_t* __restrict__ ids,
                                            const int32_t* __restrict__ chunk_base,
                                            const int32_t* __restrict__ kept,
                                            int32_t* __restrict__ offsets,
                                            int32_t* __restrict__ slot_row,
                                            int32_t* __restrict__ row_token, int positions_only,
                                            const int32_t* __restrict__ cap_base, int32_t* sm) {
  int32_t* off = sm;                       // [E+1]
  int32_t* wbase = sm + E + 1;             // [8][E]
  int32_t* s_ids = wbase + 8 * E;          // [256·k]
  __shared__ int32_t part[kDispatchThreads];
  const int tid = threadIdx.x, warp = tid >> 5;
  const int64_t chunk0 = int64_t(blockIdx.x) * kChunkTokens;
  {
    // The chunk's ids, coalesced, once.
    const int64_t n_ids = (T - chunk0 < kChunkTokens ? T - chunk0 : kChunkTokens) * k;
    const int32_t* src = ids + chunk0 * k;
    for (int i = tid; i < n_ids; i += kDispatchThreads) s_ids[i] = src[i];
  }

  // Expert offsets: exclusive scan of kept[0..E) (positions_only: the
  // per-expert capacity instead, C or C - cap_base[e]).
  if (positions_only) {
    for (int e = tid; e < E; e += kDispatchThreads) off[e] = int32_t(C - (cap_base ? cap_base[e] : 0));
  } else {
    block_exclusive_scan(E, kept, off, part);
  }
  for (int i = tid; i < 8 * E; i += kDispatchThreads) wbase[i] = 0;
  __syncthreads();
  if (blockIdx.x == 0 && !positions_only)
    for (int e = tid; e <= E; e += kDispatchThreads) offsets[e] = off[e];

  // Per-warp histograms of this chunk.
  const int64_t t_own = chunk0 + tid;
  if (t_own < T)
    for (int r = 0; r < k; ++r) {
      const int e = s_ids[tid * k + r];
      if (e >= 0 && e < E) atomicAdd(&wbase[warp * E + e], 1);
    }
  __syncthreads();
  // wbase[w][e] <- chunk base of e + counts of e in warps before w.
  for (int e = tid; e < E; e += kDispatchThreads) {
    int32_t acc = chunk_base[int64_t(blockIdx.x) * E + e];
    for (int w = 0; w < 8; ++w) {
      const int32_t v = wbase[w * E + e];
      wbase[w * E + e] = acc;
      acc += v;
    }
  }
  __syncthreads();
  walk_slots(T, E, k, C, chunk0, s_ids, wbase + warp * E, off, slot_row, row_token,
             positions_only);
}

__global__ void __launch_bounds__(kDispatchThreads)
    assign_kernel(int64_t T, int E, int k, int64_t C, const int32_t* __restrict__ ids,
                  const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ kept,
                  int32_t* __restrict__ offsets, int32_t* __restrict__ slot_row,
                  int32_t* __restrict__ row_token, int positions_only,
                  const int32_t* __restrict__ cap_base) {
  extern __shared__ int32_t sm[];
  pdl_wait();
  pdl_trigger();
  assign_body(T, E, k, C, ids, chunk_base, kept, offsets, slot_row, row_token, positions_only,
              cap_base, sm);
}

// A call with a single chunk (T <= 256, e.g. a decode step): one block does
// the whole dispatch from shared memory — ids, the warps' histograms (whose
// sum is counts and whose prefix over warps gives each warp's base; the
// single chunk's base is 0), kept, offsets, the statistics and the positions
// — so its only global round trips are the loads of ids and of the router's
// fixed-point column sums (issued together) and the stores.  Dynamic shared
// memory: off[E+1] | wbase[8][E] | ids[256·k] | counts[E] | kept[E] | psum[E].
__global__ void __launch_bounds__(kDispatchThreads)
    dispatch_small_kernel(int64_t T, int E, int k, int64_t C, const int32_t* __restrict__ ids,
                          int32_t* status, int32_t* __restrict__ counts,
                          int32_t* __restrict__ kept, AuxArgs aux,
                          int32_t* __restrict__ offsets, int32_t* __restrict__ slot_row,
                          int32_t* __restrict__ row_token) {
  extern __shared__ int32_t sm[];
  int32_t* off = sm;                                   // [E+1]
  int32_t* wbase = off + E + 1;                        // [8][E]
  int32_t* s_ids = wbase + 8 * E;                      // [256·k]
  int32_t* s_cnt = s_ids + kChunkTokens * k;           // [E]
  int32_t* s_kept = s_cnt + E;                         // [E]
  float* s_psum = reinterpret_cast<float*>(s_kept + E);  // [E]
  __shared__ int32_t part[kDispatchThreads];
  __shared__ float s_red[kAuxThreads];
  __shared__ unsigned long long s_kept_sum;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < 8 * E; i += kDispatchThreads) wbase[i] = 0;
  pdl_wait();
  pdl_trigger();
  const int64_t n_ids = T * k;
  for (int64_t i = tid; i < n_ids; i += kDispatchThreads) s_ids[i] = ids[i];
  if (aux.f) {
    // psum from the router's fixed-point column sums (as psum_from_fixed,
    // with every copy's load issued before the first add), else as given.
    for (int c = tid; c < E; c += kDispatchThreads) {
      float p;
      if (aux.psum_fixed) {
        unsigned long long v[kPsumReplicas];
#pragma unroll
        for (int r = 0; r < kPsumReplicas; ++r) v[r] = __ldcg(aux.psum_fixed + r * kPsumFixedMaxE + c);
        unsigned long long fx = 0;
#pragma unroll
        for (int r = 0; r < kPsumReplicas; ++r) fx += v[r];
#pragma unroll
        for (int r = 0; r < kPsumReplicas; ++r) __stcg(aux.psum_fixed + r * kPsumFixedMaxE + c, 0ull);
        p = float(double(fx) * kPsumFixInv);
        aux.psum[c] = p;
      } else {
        p = __ldcg(aux.psum + c);
      }
      s_psum[c] = p;
    }
  }
  __syncthreads();
  if (tid < T)
    for (int r = 0; r < k; ++r) {
      const int e = s_ids[tid * k + r];
      if (e >= 0 && e < E)
        atomicAdd(&wbase[warp * E + e], 1);
      else
        set_status(status, MOE_ERR_INVALID_ARG);
    }
  __syncthreads();
  // counts, kept, and wbase[w][e] <- counts of e in warps before w.
  for (int e = tid; e < E; e += kDispatchThreads) {
    int32_t acc = 0;
    for (int w = 0; w < 8; ++w) {
      const int32_t v = wbase[w * E + e];
      wbase[w * E + e] = acc;
      acc += v;
    }
    const int32_t kp = int32_t(acc < C ? acc : C);
    s_cnt[e] = acc;
    s_kept[e] = kp;
    counts[e] = acc;
    kept[e] = kp;
  }
  __syncthreads();
  if (aux.f)
    aux_stats_block<true>(E, T, aux.alpha, s_cnt, s_psum, aux.f, aux.pbar, aux.l_aux, s_red);
  if (aux.health) {
    __syncthreads();
    routing_health_block<true>(E, T, k, s_cnt, s_kept, aux.health, s_red, &s_kept_sum);
  }
  block_exclusive_scan(E, s_kept, off, part);
  for (int e = tid; e <= E; e += kDispatchThreads) offsets[e] = off[e];
  walk_slots(T, E, k, C, 0, s_ids, wbase + warp * E, off, slot_row, row_token, 0);
}

// T > 256 in one launch: a cooperative grid (every block resident) of one
// block per 256-token chunk plus one summary block.  Each chunk block counts
// its chunk (the warps' histograms in shared memory), publishes the chunk's
// counts and meets the others at a bounded grid barrier; then it reads all
// chunks' counts, forms kept, the expert offsets and its own chunk's base per
// expert (the counts of the chunks before it) and walks its slots.  The
// summary block (the last one) loads the router's column sums before the
// barrier, and after it writes counts, kept and offsets and runs the
// statistics, in parallel with the chunk blocks' walks.  The results are those
// of histogram_kernel + assign_kernel.  Dynamic shared memory: off[E+1] |
// wbase[8][E] | ids[256·k] | counts[E] | kept[E] | psum[E].
__global__ void __launch_bounds__(kDispatchThreads)
    dispatch_onepass_kernel(int64_t T, int E, int k, int64_t C, const int32_t* __restrict__ ids,
                            int32_t* __restrict__ chunk_counts, int32_t* status, int* bar,
                            int expect, uint64_t limit_ns, int32_t* __restrict__ counts,
                            int32_t* __restrict__ kept, AuxArgs aux,
                            int32_t* __restrict__ offsets, int32_t* __restrict__ slot_row,
                            int32_t* __restrict__ row_token) {
  extern __shared__ int32_t sm[];
  int32_t* off = sm;                                     // [E+1]
  int32_t* wbase = off + E + 1;                          // [8][E]
  int32_t* s_ids = wbase + 8 * E;                        // [256·k]
  int32_t* s_cnt = s_ids + kChunkTokens * k;             // [E]
  int32_t* s_kept = s_cnt + E;                           // [E]
  float* s_psum = reinterpret_cast<float*>(s_kept + E);  // [E]
  __shared__ int32_t part[kDispatchThreads];
  __shared__ float s_red[kAuxThreads];
  __shared__ unsigned long long s_kept_sum;
  __shared__ int s_ok;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int nb = int(gridDim.x) - 1;                     // chunk blocks
  const bool summary = int(blockIdx.x) == nb;
  const int64_t chunk0 = int64_t(blockIdx.x) * kChunkTokens;
  for (int i = tid; i < 8 * E; i += kDispatchThreads) wbase[i] = 0;
  pdl_wait();
  pdl_trigger();
  if (summary) {
    // psum from the router's fixed-point column sums (psum_from_fixed's
    // arithmetic), or as given; independent of the counts, so before the
    // barrier.
    if (aux.f)
      for (int c = tid; c < E; c += kDispatchThreads) {
        float pv;
        if (aux.psum_fixed) {
          unsigned long long fx = 0;
#pragma unroll 8
          for (int r = 0; r < kPsumReplicas; ++r) fx += __ldcg(aux.psum_fixed + r * kPsumFixedMaxE + c);
#pragma unroll 8
          for (int r = 0; r < kPsumReplicas; ++r) __stcg(aux.psum_fixed + r * kPsumFixedMaxE + c, 0ull);
          pv = float(double(fx) * kPsumFixInv);
          aux.psum[c] = pv;
        } else {
          pv = __ldcg(aux.psum + c);
        }
        s_psum[c] = pv;
      }
  } else {
    const int64_t n_tok = T - chunk0 < kChunkTokens ? T - chunk0 : kChunkTokens;
    for (int64_t i = tid; i < n_tok * k; i += kDispatchThreads) s_ids[i] = ids[chunk0 * k + i];
    __syncthreads();
    if (tid < n_tok)
      for (int r = 0; r < k; ++r) {
        const int e = s_ids[tid * k + r];
        if (e >= 0 && e < E)
          atomicAdd(&wbase[warp * E + e], 1);
        else
          set_status(status, MOE_ERR_INVALID_ARG);
      }
    __syncthreads();
    // wbase[w][e] <- counts of e in warps before w; the chunk's count of e.
    for (int e = tid; e < E; e += kDispatchThreads) {
      int32_t acc = 0;
      for (int w = 0; w < 8; ++w) {
        const int32_t v = wbase[w * E + e];
        wbase[w * E + e] = acc;
        acc += v;
      }
      __stcg(chunk_counts + int64_t(blockIdx.x) * E + e, acc);
    }
  }
  if (grid_barrier_wait(bar, expect, status, limit_ns, &s_ok)) {
    // Every chunk's counts: the totals, and (chunk blocks) this chunk's base
    // per expert.
    for (int e = tid; e < E; e += kDispatchThreads) {
      int32_t tot = 0, base = 0;
#pragma unroll 8
      for (int b = 0; b < nb; ++b) {
        const int32_t v = __ldcg(chunk_counts + int64_t(b) * E + e);
        base += b < int(blockIdx.x) ? v : 0;
        tot += v;
      }
      const int32_t kp = int32_t(tot < C ? tot : C);
      s_cnt[e] = tot;
      s_kept[e] = kp;
      if (summary) {
        counts[e] = tot;
        kept[e] = kp;
      } else {
        for (int w = 0; w < 8; ++w) wbase[w * E + e] += base;
      }
    }
    __syncthreads();
    block_exclusive_scan(E, s_kept, off, part);
    if (summary) {
      for (int e = tid; e <= E; e += kDispatchThreads) offsets[e] = off[e];
      if (aux.f)
        aux_stats_block<true>(E, T, aux.alpha, s_cnt, s_psum, aux.f, aux.pbar, aux.l_aux, s_red);
      if (aux.health) {
        __syncthreads();
        routing_health_block<true>(E, T, k, s_cnt, s_kept, aux.health, s_red, &s_kept_sum);
      }
    } else {
      walk_slots(T, E, k, C, chunk0, s_ids, wbase + warp * E, off, slot_row, row_token, 0);
    }
  }
  grid_barrier_depart(bar);
}

// Overflow reroute, step 2: the m-th slot of token t that the first fill
// dropped (pos0 < 0), in rank order, is offered to cand[t*k + m]; other slots
// offer nothing (-1).  One thread per token.
__global__ void __launch_bounds__(256)
    reroute_offer_kernel(int64_t T, int k, const int32_t* __restrict__ pos0,
                         const int32_t* __restrict__ cand, int32_t* __restrict__ ids1) {
  pdl_wait();
  pdl_trigger();
  for (int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; t < T;
       t += int64_t(gridDim.x) * blockDim.x) {
    int m = 0;
    for (int r = 0; r < k; ++r) {
      int32_t e = -1;
      if (pos0[t * k + r] < 0) {
        e = cand[t * k + m];
        ++m;
      }
      ids1[t * k + r] = e;
    }
  }
}

// Overflow reroute, last step: offsets = exclusive scan of the final kept;
// a slot kept by the first fill sits at offsets[e] + pos0, a served offer at
// offsets[e'] + kept0[e'] + pos1 (after the expert's own rows); row_token for
// every kept row.  Every block forms the offsets in shared memory; block 0
// writes them.
__global__ void __launch_bounds__(kDispatchThreads)
    reroute_finalize_kernel(int64_t T, int E, int k, const int32_t* __restrict__ ids,
                            const int32_t* __restrict__ ids1, const int32_t* __restrict__ pos0,
                            const int32_t* __restrict__ pos1, const int32_t* __restrict__ kept0,
                            const int32_t* __restrict__ kept, int32_t* __restrict__ offsets,
                            int32_t* __restrict__ slot_row, int32_t* __restrict__ row_token) {
  extern __shared__ int32_t off[];  // [E+1]
  __shared__ int32_t part[kDispatchThreads / 32];
  pdl_wait();
  pdl_trigger();
  block_exclusive_scan(E, kept, off, part);
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = off[e];
  const int64_t n = T * k;
  for (int64_t s = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; s < n;
       s += int64_t(gridDim.x) * blockDim.x) {
    int32_t row = -1;
    if (pos0[s] >= 0) {
      row = off[ids[s]] + pos0[s];
    } else if (pos1[s] >= 0) {
      const int32_t e = ids1[s];
      row = off[e] + kept0[e] + pos1[s];
    }
    slot_row[s] = row;
    if (row >= 0) row_token[row] = int32_t(s / k);
  }
}

// xd[slot_row[t,r]] = x[t] for every kept slot; one warp per token, the row
// is read once (16-byte vectors, 4 in flight per lane) and written k times.
__global__ void __launch_bounds__(256)
    scatter_rows_kernel(int64_t T, int k, int64_t row_vecs, int64_t n_parts, int64_t part_vecs,
                        const uint4* __restrict__ x, const int32_t* __restrict__ slot_row,
                        uint4* __restrict__ xd) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  pdl_wait();
  pdl_trigger();
  for (int64_t it = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       it < T * n_parts; it += warps) {
    const int64_t t = it / n_parts;
    const int64_t vb = (it % n_parts) * part_vecs;
    const int64_t ve = vb + part_vecs < row_vecs ? vb + part_vecs : row_vecs;
    const int32_t my_row = lane < k ? slot_row[t * k + lane] : -1;
    const unsigned kept_mask = __ballot_sync(0xffffffffu, my_row >= 0);
    if (kept_mask == 0) continue;
    const uint4* src = x + t * row_vecs;
    for (int64_t v0 = vb; v0 < ve; v0 += 4 * 32) {
      uint4 buf[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t v = v0 + u * 32 + lane;
        if (v < ve) buf[u] = __ldcs(src + v);
      }
      unsigned m = kept_mask;
      while (m) {
        const int r = __ffs(m) - 1;
        m &= m - 1;
        const int32_t row = __shfl_sync(0xffffffffu, my_row, r);
        uint4* dst = xd + int64_t(row) * row_vecs;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t v = v0 + u * 32 + lane;
          if (v < ve) dst[v] = buf[u];
        }
      }
    }
  }
}

// The one-pass dispatch (dispatch_onepass_kernel) when every chunk's block
// can be resident at once (MOE_DISPATCH_ONEPASS=0 turns it off, a
// cross-check in tests).
constexpr uint64_t kGridBarrierLimitNs = 4000000000ull;  // 4 s
bool onepass_fits(const moe_config_t& c, int64_t n_chunks) {
  const char* v = std::getenv("MOE_DISPATCH_ONEPASS");
  if (v && std::strcmp(v, "0") == 0) return false;
  const size_t smem = size_t(c.E + 1 + 8 * c.E + kChunkTokens * c.k + 3 * c.E) * 4;
  if (ensure_dynamic_smem(reinterpret_cast<const void*>(dispatch_onepass_kernel), smem) !=
      cudaSuccess)
    return false;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_onepass_kernel,
                                                    kDispatchThreads, smem) != cudaSuccess)
    return false;
  return n_chunks + 1 <= int64_t(per_sm) * device_sms();
}

cudaError_t launch_dispatch(const moe_config_t& c, int64_t C, const void* x,
                            const int32_t* ids, int32_t* counts, int32_t* kept,
                            int32_t* offsets, int32_t* slot_row, int32_t* row_token, void* xd,
                            int32_t* chunk_counts, int32_t* status, int* counter, int* grid_bar,
                            const AuxArgs* aux, const RerouteBufs* rr, cudaStream_t st) {
  if (rr && !counter) return cudaErrorInvalidValue;
  const int64_t n_chunks = (c.T + kChunkTokens - 1) / kChunkTokens;
  const AuxArgs no_aux{0.f, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  const AuxArgs aux_v = (aux && counter) ? *aux : no_aux;
  const size_t hist_smem = size_t(c.E) * 4;
  const size_t assign_smem = size_t(c.E + 1 + 8 * c.E + kChunkTokens * c.k) * 4;
  cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(assign_kernel), assign_smem);
  if (err != cudaSuccess) return err;
  auto histogram = [&](const int32_t* ids_, int32_t* counts_, int32_t* kept_, const AuxArgs& a,
                       int skip_neg, const int32_t* cap_base) {
    cudaError_t e = launch_pdl(histogram_kernel, dim3(unsigned(n_chunks)), dim3(kDispatchThreads),
                               hist_smem, st, c.T, c.E, c.k, ids_, chunk_counts, status, counter,
                               C, counts_, kept_, a, skip_neg, cap_base);
    count_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
  };
  auto assign = [&](const int32_t* ids_, const int32_t* kept_, int32_t* slot_row_,
                    int positions_only, const int32_t* cap_base) {
    cudaError_t e = launch_pdl(assign_kernel, dim3(unsigned(n_chunks)), dim3(kDispatchThreads),
                               assign_smem, st, c.T, c.E, c.k, C, ids_,
                               static_cast<const int32_t*>(chunk_counts), kept_, offsets,
                               slot_row_, row_token, positions_only, cap_base);
    count_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
  };
  if (!rr && n_chunks == 1) {
    const size_t small_smem = assign_smem + size_t(3 * c.E) * 4;
    err = ensure_dynamic_smem(reinterpret_cast<const void*>(dispatch_small_kernel), small_smem);
    if (err != cudaSuccess) return err;
    err = launch_pdl(dispatch_small_kernel, dim3(1), dim3(kDispatchThreads), small_smem, st, c.T,
                     c.E, c.k, C, ids, status, counts, kept, aux_v, offsets, slot_row,
                     row_token);
    count_launch();
    if (err != cudaSuccess || (err = cudaGetLastError()) != cudaSuccess) return err;
  } else if (!rr && grid_bar && counter && onepass_fits(c, n_chunks)) {
    const size_t smem = assign_smem + size_t(3 * c.E) * 4;
    err = ensure_dynamic_smem(reinterpret_cast<const void*>(dispatch_onepass_kernel), smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(n_chunks + 1));  // the chunks and the summary block
    cfg.blockDim = dim3(kDispatchThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;  // every block resident: the grid barrier
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    err = cudaLaunchKernelEx(&cfg, dispatch_onepass_kernel, c.T, c.E, c.k, C, ids, chunk_counts,
                             status, grid_bar, int(n_chunks + 1), kGridBarrierLimitNs, counts, kept,
                             aux_v, offsets, slot_row, row_token);
    count_launch();
    if (err != cudaSuccess || (err = cudaGetLastError()) != cudaSuccess) return err;
  } else if (!rr) {
    if ((err = histogram(ids, counts, kept, aux_v, 0, nullptr)) != cudaSuccess) return err;
    if (!counter) {
      expert_scan_kernel<<<unsigned(c.E), 256, 0, st>>>(n_chunks, c.E, C, chunk_counts, counts,
                                                         kept);
      count_launch();
      if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    if ((err = assign(ids, kept, slot_row, 0, nullptr)) != cudaSuccess) return err;
  } else {
    // [MoE 模型原理 §4.3] reroute: first fill (positions only), offers to the
    // next candidates, second fill into the room left, final rows.
    if ((err = histogram(ids, counts, rr->kept0, no_aux, 0, nullptr)) != cudaSuccess) return err;
    if ((err = assign(ids, nullptr, rr->pos0, 1, nullptr)) != cudaSuccess) return err;
    const int64_t tb = (c.T + 255) / 256;
    err = launch_pdl(reroute_offer_kernel, dim3(unsigned(tb < 4096 ? tb : 4096)), dim3(256), 0,
                     st, c.T, c.k, static_cast<const int32_t*>(rr->pos0), rr->cand, rr->ids1);
    count_launch();
    if (err != cudaSuccess || (err = cudaGetLastError()) != cudaSuccess) return err;
    AuxArgs a1 = aux_v;
    a1.counts_f = counts;  // f and health use the first choices' counts
    err = histogram(rr->ids1, rr->counts1, kept, a1, 1, rr->kept0);
    if (err != cudaSuccess) return err;
    if ((err = assign(rr->ids1, nullptr, rr->pos1, 1, rr->kept0)) != cudaSuccess) return err;
    const int64_t sb = (c.T * c.k + kDispatchThreads - 1) / kDispatchThreads;
    const size_t fsmem = size_t(c.E + 1) * 4;
    err = ensure_dynamic_smem(reinterpret_cast<const void*>(reroute_finalize_kernel), fsmem);
    if (err != cudaSuccess) return err;
    err = launch_pdl(reroute_finalize_kernel, dim3(unsigned(sb < 2048 ? sb : 2048)),
                     dim3(kDispatchThreads), fsmem, st, c.T, c.E, c.k, ids,
                     static_cast<const int32_t*>(rr->ids1), static_cast<const int32_t*>(rr->pos0),
                     static_cast<const int32_t*>(rr->pos1),
                     static_cast<const int32_t*>(rr->kept0), static_cast<const int32_t*>(kept),
                     offsets, slot_row, row_token);
    count_launch();
    if (err != cudaSuccess || (err = cudaGetLastError()) != cudaSuccess) return err;
  }
  if (!xd) return cudaSuccess;  // the first GEMM gathers the rows itself
  const int elem = c.dtype == MOE_DT_BF16 ? 2 : 4;
  const int64_t row_vecs = int64_t(c.d) * elem / 16;
  const RowSplit rs = row_split(c.T, row_vecs, 128);
  const int sms = device_sms();
  const int64_t want = (c.T * rs.n_parts + 7) / 8;
  const unsigned grid = unsigned(want < int64_t(sms) * 8 ? want : int64_t(sms) * 8);
  err = launch_pdl(scatter_rows_kernel, dim3(grid), dim3(256), 0, st, c.T, c.k, row_vecs,
                   rs.n_parts, rs.part_vecs, static_cast<const uint4*>(x), slot_row,
                   static_cast<uint4*>(xd));
  count_launch();
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace moe
