/*
 * moe.h — C ABI of libmoe.so: the forward pass of one Mixture-of-Experts
 * layer on one NVIDIA B300 (sm_103a).
 *
 * The layer follows "MoE 模型原理：路由、专家负载、容量、通信与推理成本"
 * (wrblog.cn), cited below as [MoE 模型原理 §n]:
 *
 *   route    §2.1–§2.2  s_t = W_r x_t + b_r, p_t = softmax(s_t),
 *                       S_t = TopK(p_t, k), weights p̃ (optionally renormalised)
 *   dispatch §4.1–§4.3, §5  capacity C = ceil(c·T·k/E); slots take expert
 *                       positions first come in (token, rank) order; overflow
 *                       is dropped; kept rows are packed expert by expert
 *   experts  §1         E_i(x) = W2 σ(W1 x + b1) + b2, as grouped GEMMs over
 *                       the ragged per-expert row ranges
 *   combine  §2.2, §5   y_t = Σ_{kept r} p̃_{t,r} E_{S_t[r]}(x_t), token order
 *   aux      §3.2       f_i = counts_i/T, p̄_i = Σ_t p_{t,i}/T,
 *                       L_aux = α·E·Σ_i f_i p̄_i
 *
 * Conventions for every call:
 *  - Pointers named as tensors are DEVICE pointers to caller-owned memory;
 *    `cfg`, `status` and `bytes` are host pointers.  The library never
 *    allocates device memory and never synchronises the stream; every call
 *    only enqueues kernels on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and returns.
 *  - Layouts are dense row-major.  "act" tensors (x, xd, H, yd, y, and the
 *    weights W_r, W1, W2) have element type cfg->dtype: MOE_DT_F32 (fp32) or
 *    MOE_DT_BF16 (bf16).  Biases, logits, weights of the combine, psum and
 *    the statistics are fp32; ids, counts and indices are int32.
 *  - Sizes that depend on the routing stay on the device: offsets[E] is the
 *    number of kept rows; rows at or beyond it in xd, H, yd are not written.
 *  - Synchronous errors (returned): MOE_ERR_INVALID_ARG for a NULL tensor or
 *    a shape outside the limits below; MOE_ERR_UNSUPPORTED for an unbuilt
 *    combination; MOE_ERR_WORKSPACE if ws_bytes < moe_workspace_size();
 *    MOE_ERR_CUDA if a launch fails.  moe_last_error() gives a message.
 *  - Asynchronous errors: kernels record the first error code in a status
 *    word inside the workspace (an out-of-range expert id -> INVALID_ARG; a
 *    bounded wait that gave up -> TIMEOUT).  Read it with
 *    moe_get_device_status() after synchronising.
 *  - Limits: T >= 1, T*k < 2^31; 1 <= k <= 16; k <= E <= 1024; d and d_ff
 *    multiples of 8 (rows are moved as 16-byte vectors); 2^-30 <= c <= 2^30.
 *  - NaN or Inf inputs give unspecified results.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t moe_status_t;
enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,
  MOE_ERR_UNSUPPORTED = 2,
  MOE_ERR_CUDA = 3,
  MOE_ERR_WORKSPACE = 4,
  MOE_ERR_TIMEOUT = 5
};

enum { MOE_DT_F32 = 0, MOE_DT_BF16 = 1 };
enum { MOE_ACT_RELU = 0, MOE_ACT_GELU_TANH = 1 };

/* Layer configuration; plain fields so any FFI can build it. */
typedef struct moe_config {
  int64_t T;                /* tokens in this call (the capacity group, §4.1) */
  int32_t d;                /* model width */
  int32_t d_ff;             /* expert hidden width */
  int32_t E;                /* experts */
  int32_t k;                /* experts per token */
  double capacity_factor;   /* c in C = ceil(c·T·k/E) */
  int32_t renormalize;      /* 1: p̃ = p/Σ_{S_t} p (§2.2); 0: raw p */
  int32_t act;              /* MOE_ACT_* : σ of the expert FFN */
  int32_t dtype;            /* MOE_DT_* : x, weights, xd, H, yd, y */
  int32_t write_logits;     /* 1: moe_route also writes fp32 logits[T,E] */
  int32_t reroute;          /* 1: overflow goes to the next candidate (§4.3) */
  int32_t fuse_dispatch;    /* 1: no xd; the first GEMM gathers x rows (moe_ffn_up_gather) */
  int32_t fuse_combine;     /* 1: the second GEMM also combines (moe_ffn_down_combine) */
} moe_config_t;

/* Every tensor of one forward pass (all device pointers). */
typedef struct moe_tensors {
  /* inputs */
  const void* x;        /* [T, d]                                     */
  const void* Wr;       /* [E, d]      router, row i scores expert i  */
  const float* br;      /* [E]         router bias                    */
  const void* W1;       /* [E, d_ff, d]  maps d -> d_ff               */
  const float* b1;      /* [E, d_ff]                                  */
  const void* W2;       /* [E, d, d_ff]  maps d_ff -> d               */
  const float* b2;      /* [E, d]                                     */
  /* routing outputs */
  float* logits;        /* [T, E]  written only if cfg->write_logits  */
  int32_t* topk_ids;    /* [T, k]  descending score, ties to lower id */
  float* topk_w;        /* [T, k]  combine weights p̃                  */
  float* psum;          /* [E]     Σ_t p_{t,i}                         */
  /* dispatch outputs */
  int32_t* counts;      /* [E]     slots routed to expert (pre-capacity) */
  int32_t* kept;        /* [E]     min(counts, C)                     */
  int32_t* offsets;     /* [E+1]   exclusive scan of kept             */
  int32_t* slot_row;    /* [T, k]  row in xd of slot (t,r), -1 if dropped */
  int32_t* row_token;   /* [R]     token of each kept row, R = moe_max_rows() */
  void* xd;             /* [R, d]  per-expert contiguous token rows   */
  /* expert outputs */
  void* H;              /* [R, d_ff] hidden activations σ(W1 x + b1)  */
  void* yd;             /* [R, d]    expert outputs                   */
  /* layer outputs */
  void* y;              /* [T, d]  combined output (no residual add)  */
  float* f;             /* [E]     f_i                                */
  float* pbar;          /* [E]     p̄_i                                */
  float* l_aux;         /* [1]     L_aux                              */
  /* optional inputs/outputs (NULL: not used) */
  const float* sel_bias; /* [E] expert bias for the top-k choice only (moe_route_sel) */
  float* health;         /* [4] routing-health indicators (moe_routing_health) */
} moe_tensors_t;

/* [MoE 模型原理 §4.1] Capacity C = ceil(c·T·k/E), exact for the binary value
 * of c.  Host only, pure.  Returns -1 if cfg is invalid. */
int64_t moe_capacity(const moe_config_t* cfg);

/* Rows of the dispatch buffer to allocate: min(T·k, E·C).  -1 if invalid. */
int64_t moe_max_rows(const moe_config_t* cfg);

/* Bytes of scratch workspace the stage calls need (272 KiB header with the
 * status word, completion counters and the router's fixed-point column-sum
 * accumulators; per-chunk histograms; per-block probability partial sums; the
 * tensor-core router's fp32 partial logits, nsplit·T·E floats, nsplit > 1 only
 * for small T; with cfg->reroute the reroute's [T, k] arrays; with
 * cfg->fuse_combine the combine's arrival counters, 2 int32 per token and
 * 256-wide column tile of d).  Host only.  A workspace serves one stream at a
 * time. */
moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes);

/* Clear the whole workspace (ws_bytes bytes, at least the 272 KiB header):
 * the device status word, the counters the kernels use to find the last
 * block of a grid and the column-sum accumulators (enqueued on stream;
 * kernels leave them at zero).  Call once after allocating a workspace, and
 * after reading a nonzero status. */
moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* [MoE 模型原理 §2.1–§2.2] Router: logits s = x W_rᵀ + b_r (fp32 accumulate),
 * softmax, top-k with ties to the lower expert index, combine weights
 * (renormalised over the selected set iff cfg->renormalize), and the column
 * sums psum[i] = Σ_t p_{t,i}, deterministic: per-block partial sums in a
 * fixed order (each p_{t,i} rounded to 31 fraction bits first with the
 * tensor-core router), added exactly as 64-bit fixed-point integers.  logits may be NULL unless cfg->write_logits.
 * With cfg->reroute it also leaves each token's next candidates (the experts
 * ranked k .. 2k-1) in the workspace for moe_dispatch. */
moe_status_t moe_route(const moe_config_t* cfg, const void* x, const void* Wr, const float* br,
                       float* logits, int32_t* topk_ids, float* topk_w, float* psum, void* ws,
                       size_t ws_bytes, void* stream);

/* [MoE 模型原理 §4.1–§4.3, §5] Histogram, capacity, first-come positions in
 * (token, rank) order, and the permutation xd[slot_row[t,r]] = x[t] for
 * every kept slot.  Writes counts, kept, offsets, slot_row, row_token, xd.
 * With cfg->reroute (§4.3, second policy) an overflowing slot is then offered
 * to its token's next candidate (the m-th overflowing slot of a token, in
 * rank order, to the expert ranked k + m, read from the candidates the last
 * moe_route call left in this workspace); offers are served first come in
 * (token, rank) order into the room each expert has left, and an expert's
 * rerouted rows follow its own.  counts stay the first choices' (f_i is over
 * S_t); kept, offsets, slot_row and row_token are final; a rerouted slot keeps
 * its combine weight.
 * With cfg->fuse_dispatch no row is copied: xd may be NULL and is not
 * written (moe_ffn_up_gather reads the rows from x).
 * topk_ids need not be distinct within a token: every (t, r) is its own
 * slot, and slots of one token that name the same expert take consecutive
 * positions in rank order.  An id outside [0, E) names no expert: that slot
 * is not counted, its slot_row is -1, and the workspace status word receives
 * MOE_ERR_INVALID_ARG; every other slot is dispatched as if it were absent. */
moe_status_t moe_dispatch(const moe_config_t* cfg, const void* x, const int32_t* topk_ids,
                          int32_t* counts, int32_t* kept, int32_t* offsets, int32_t* slot_row,
                          int32_t* row_token, void* xd, void* ws, size_t ws_bytes, void* stream);

/* The dispatch stage for callers that cannot allocate device memory (for
 * example a plugin inside a host framework whose memory pool owns the whole
 * device, or a latency-critical path that may not take cudaMalloc's implicit
 * synchronisation), so cannot provide the workspace moe_dispatch needs.
 * This call has no counterpart in the paper: it is an interface choice.
 * Same outputs as moe_dispatch; the per-chunk histogram lives in a fixed
 * 1 MiB device array inside the library (held by every GPU that loads the
 * library until exit), so this call allocates nothing.
 *  - requires ceil(T/256)·E <= 262144, else MOE_ERR_INVALID_ARG (no launch);
 *  - status: optional device int32 (may be NULL) that receives
 *    MOE_ERR_INVALID_ARG if an expert id is out of range; the caller zeroes
 *    it; it is written only on error;
 *  - all calls on a device share the array: calls that overlap on the GPU
 *    race; calls ordered on one stream do not (nothing carries over);
 *  - the first call on each device looks up the array's address; make that
 *    call before any stream capture. */
moe_status_t moe_dispatch_noalloc(const moe_config_t* cfg, const void* x,
                                  const int32_t* topk_ids, int32_t* counts, int32_t* kept,
                                  int32_t* offsets, int32_t* slot_row, int32_t* row_token,
                                  void* xd, int32_t* status, void* stream);

/* [MoE 模型原理 §1] First expert GEMM over the ragged groups given by
 * offsets: H[rows of e] = σ(xd[rows of e] W1[e]ᵀ + b1[e]).
 * Ordering: the GEMM kernels are launched with programmatic dependent launch.
 * The kernel reads offsets (and, with at most 64 rows per expert, starts
 * copying weights) as soon as it is scheduled, which can be before the
 * previous kernel in the stream has finished (it still waits for that kernel
 * before reading xd).  So offsets must be complete when the kernel just
 * before this call in the stream starts, or be written by a kernel that does
 * not signal its dependents early (griddepcontrol.launch_dependents) or by a
 * copy.  moe_dispatch ends with the row scatter, which starts only after the
 * kernel that writes offsets has finished, and every kernel of this library
 * waits for its predecessor before it signals: moe_dispatch → moe_ffn_up →
 * moe_ffn_down meets the condition.  The same holds for moe_ffn_down (which
 * waits before reading H). */
moe_status_t moe_ffn_up(const moe_config_t* cfg, const void* xd, const int32_t* offsets,
                        const void* W1, const float* b1, void* H, void* ws, size_t ws_bytes,
                        void* stream);

/* moe_ffn_up with the permutation folded into the GEMM's operand load (the
 * fused permutation/dispatch kernel of [MoE Gate 分布式通信 mianshidashi,
 * 06]): H[row] = σ(x[row_token[row]] W1[e]ᵀ + b1[e]) for the rows of each
 * expert e, so the dispatch buffer xd is neither written nor read.  Same
 * result, bit for bit, as moe_ffn_up on the xd that moe_dispatch would write.
 *  - x [T, d] and row_token (from moe_dispatch) are device pointers; x, W1
 *    and H 16-byte aligned; a row_token entry outside [0, T) reads as a zero
 *    row;
 *  - bf16 layers on the tensor-core GEMM only: MOE_ERR_UNSUPPORTED (no
 *    launch) for fp32 layers and for layers with at most 64 rows per expert
 *    (min(C, T·k) <= 64, the swapped decode GEMM). */
moe_status_t moe_ffn_up_gather(const moe_config_t* cfg, const void* x, const int32_t* row_token,
                               const int32_t* offsets, const void* W1, const float* b1, void* H,
                               void* ws, size_t ws_bytes, void* stream);

/* [MoE 模型原理 §1] Second expert GEMM: yd[rows of e] = H W2[e]ᵀ + b2[e]. */
moe_status_t moe_ffn_down(const moe_config_t* cfg, const void* H, const int32_t* offsets,
                          const void* W2, const float* b2, void* yd, void* ws, size_t ws_bytes,
                          void* stream);

/* moe_ffn_down with the combine folded into the GEMM's epilogue (the fused
 * combine of [MoE Gate 分布式通信 mianshidashi, 06]; [MoE 模型原理 §2.2, §5]):
 * writes yd as moe_ffn_down does and y as moe_combine would from it, bit for
 * bit.  A token's k rows are finished by different CTAs: a first small
 * kernel sets a counter per token and column range of the workspace to the
 * token's number of kept slots (and writes y = 0 for a token with none);
 * each epilogue warp takes one count off per row it stored, and the warp
 * whose decrement reaches zero sums the token's k rows of that range in rank
 * order in fp32; no block waits on another.
 *  - row_token, slot_row (from moe_dispatch) and topk_w (from moe_route) are
 *    device pointers; H, W2, yd and y 16-byte aligned;
 *  - cfg->fuse_combine must be 1 (MOE_ERR_INVALID_ARG otherwise: the
 *    workspace then has no counters);
 *  - bf16 layers on the tensor-core GEMM only: MOE_ERR_UNSUPPORTED (no
 *    launch) for fp32 layers and for min(C, T·k) <= 64. */
moe_status_t moe_ffn_down_combine(const moe_config_t* cfg, const void* H, const int32_t* offsets,
                                  const int32_t* row_token, const int32_t* slot_row,
                                  const float* topk_w, const void* W2, const float* b2, void* yd,
                                  void* y, void* ws, size_t ws_bytes, void* stream);

/* moe_ffn_up followed by moe_ffn_down. */
moe_status_t moe_expert_ffn(const moe_config_t* cfg, const void* xd, const int32_t* offsets,
                            const void* W1, const float* b1, const void* W2, const float* b2,
                            void* H, void* yd, void* ws, size_t ws_bytes, void* stream);

/* [MoE 模型原理 §2.2, §5] y[t] = Σ_{r: slot_row[t,r] >= 0} topk_w[t,r]·yd[slot_row[t,r]],
 * summed in rank order in fp32; 0 for a token whose slots were all dropped.
 * Deterministic (no atomics). */
moe_status_t moe_combine(const moe_config_t* cfg, const void* yd, const int32_t* slot_row,
                         const float* topk_w, void* y, void* stream);

/* moe_route with an expert bias that moves only the choice of S_t (the
 * expert-bias routing of [EP 工程 ai-master, 一、负载均衡], which replaces the
 * auxiliary loss): experts are ranked by the fp32 sum s_{t,i} + sel_bias[i]
 * (ties to the lower index); topk_w, psum and the logits stay those of the
 * unbiased scores.  sel_bias: [E] fp32 device, or NULL (= moe_route). */
moe_status_t moe_route_sel(const moe_config_t* cfg, const void* x, const void* Wr,
                           const float* br, const float* sel_bias, float* logits,
                           int32_t* topk_ids, float* topk_w, float* psum, void* ws,
                           size_t ws_bytes, void* stream);

/* [EP 工程 ai-master, 追问 2; MoE 模型原理 §10.4] Routing-health indicators
 * from counts (before capacity) and kept (after), into health[4] (fp32,
 * device):
 *   health[0] = -Σ_i q_i ln q_i, q_i = counts_i/(T·k)  (activation entropy, nats)
 *   health[1] = (1/E) Σ_i (counts_i - T·k/E)^2       (variance of routed slots)
 *   health[2] = (1/E) Σ_i (kept_i - mean kept)^2     (variance of processed rows)
 *   health[3] = 1 - Σ_i kept_i/(T·k)                 (fraction of slots dropped)
 * One block, fixed reduction order (deterministic). */
moe_status_t moe_routing_health(const moe_config_t* cfg, const int32_t* counts,
                                const int32_t* kept, float* health, void* stream);

/* [MoE 模型原理 §3.2] f = counts/T, p̄ = psum/T, L_aux = α·E·Σ f·p̄. */
moe_status_t moe_aux_stats(const moe_config_t* cfg, const int32_t* counts, const float* psum,
                           float alpha, float* f, float* pbar, float* l_aux, void* stream);

/* The whole layer: route, dispatch, expert FFN, combine, aux (the aux
 * statistics are computed inside the dispatch launches here, with the same
 * arithmetic and results as moe_aux_stats; psum is also formed there from the
 * router's fixed-point column sums).  t->sel_bias (optional) routes as
 * moe_route_sel; t->health (optional) receives moe_routing_health's
 * indicators, computed in the same dispatch launch.  With cfg->fuse_dispatch
 * t->xd may be NULL: the dispatch writes positions and row_token only and
 * the first GEMM runs as moe_ffn_up_gather (MOE_ERR_UNSUPPORTED, before any
 * launch, where that call is unsupported); every other output is identical.
 * With cfg->fuse_combine the second GEMM runs as moe_ffn_down_combine and
 * there is no separate combine launch (same y, bit for bit; same
 * MOE_ERR_UNSUPPORTED rule).
 * If it returns an error after the router was enqueued, call
 * moe_workspace_init before the next call on that workspace. */
moe_status_t moe_forward(const moe_config_t* cfg, const moe_tensors_t* t, float alpha, void* ws,
                         size_t ws_bytes, void* stream);

/* Self-test of the bounded waits every kernel uses: one block waits on an
 * mbarrier that nothing signals, gives up after limit_ns nanoseconds (the
 * kernels' own limit is 4 s; 1e6 <= limit_ns <= 4e9) and records
 * MOE_ERR_TIMEOUT in the workspace status word, then returns.  Read it with
 * moe_get_device_status; moe_workspace_init clears it.  For tests. */
moe_status_t moe_selftest_wait_timeout(void* ws, size_t ws_bytes, int64_t limit_ns,
                                       void* stream);

/* Self-test of the one-pass dispatch's grid barrier (moe_dispatch with
 * T > 256 and no reroute runs one cooperative grid whose blocks meet at a
 * barrier in the workspace header): two blocks wait for three arrivals, give
 * up after limit_ns nanoseconds (1e6 <= limit_ns <= 4e9; the dispatch's own
 * limit is 4 s), record MOE_ERR_TIMEOUT in the workspace status word and
 * return; the barrier's counters return to zero.  For tests. */
moe_status_t moe_selftest_grid_barrier_timeout(void* ws, size_t ws_bytes, int64_t limit_ns,
                                               void* stream);

/* Read the workspace's device status word (a blocking copy; call after the
 * stream that used ws has been synchronised).  *status is MOE_OK or the
 * first asynchronous error recorded. */
moe_status_t moe_get_device_status(const void* ws, int32_t* status);

/* Kernel launches this library has issued since load (all threads). */
int64_t moe_launch_count(void);

const char* moe_status_string(moe_status_t s);

/* Message for the last synchronous error on the calling thread ("" if none). */
const char* moe_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
