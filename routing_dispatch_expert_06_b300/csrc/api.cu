// C ABI of libmoe.so: argument checks, workspace layout, and the order of the
// kernel launches for each stage.  See include/moe.h for the contract.
#include <atomic>
#include <cmath>
#include <map>
#include <mutex>
#include <tuple>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

static std::atomic<int64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static thread_local std::string g_last_error;

static moe_status_t fail(moe_status_t code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

moe_status_t report_error(moe_status_t code, const char* msg) { return fail(code, msg); }

StageRange::StageRange(const char* name) { nvtxRangePushA(name); }
StageRange::~StageRange() { nvtxRangePop(); }

namespace {
constexpr int kMaxDev = 64;
std::mutex g_cache_mu;
int g_sms[kMaxDev] = {};
int g_smem_optin[kMaxDev] = {};
std::map<const void*, size_t> g_static_smem;
std::map<std::pair<int, const void*>, size_t> g_dyn_smem;
std::map<std::tuple<int, const void*, size_t, unsigned>, int> g_clusters;

int current_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev < 0 || dev >= kMaxDev ? 0 : dev;
}
}  // namespace

int device_sms() {
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(g_cache_mu);
  if (!g_sms[dev] && cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev) !=
                         cudaSuccess)
    g_sms[dev] = 0;
  return g_sms[dev] > 0 ? g_sms[dev] : 148;
}

int device_smem_optin() {
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(g_cache_mu);
  if (!g_smem_optin[dev] &&
      cudaDeviceGetAttribute(&g_smem_optin[dev], cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
          cudaSuccess)
    g_smem_optin[dev] = 0;
  return g_smem_optin[dev];
}

size_t kernel_static_smem(const void* kernel) {
  std::lock_guard<std::mutex> lock(g_cache_mu);
  auto it = g_static_smem.find(kernel);
  if (it != g_static_smem.end()) return it->second;
  cudaFuncAttributes fa{};
  const size_t v = cudaFuncGetAttributes(&fa, kernel) == cudaSuccess ? fa.sharedSizeBytes : 0;
  g_static_smem[kernel] = v;
  return v;
}

cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes) {
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(g_cache_mu);
  size_t& have = g_dyn_smem[{dev, kernel}];
  if (have >= bytes) return cudaSuccess;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
  if (e == cudaSuccess) have = bytes;
  return e;
}

cudaError_t max_active_clusters(const void* kernel, const cudaLaunchConfig_t& cfg, int* clusters) {
  const int dev = current_device();
  unsigned csize = 1;
  for (unsigned i = 0; i < cfg.numAttrs; ++i)
    if (cfg.attrs[i].id == cudaLaunchAttributeClusterDimension) csize = cfg.attrs[i].val.clusterDim.x;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  const auto key = std::make_tuple(dev, kernel, cfg.dynamicSmemBytes, csize);
  auto it = g_clusters.find(key);
  if (it != g_clusters.end()) {
    *clusters = it->second;
    return cudaSuccess;
  }
  cudaError_t e = cudaOccupancyMaxActiveClusters(clusters, kernel, &cfg);
  if (e == cudaSuccess) g_clusters[key] = *clusters;
  return e;
}

static moe_status_t cuda_fail(cudaError_t e, const char* where) {
  return fail(MOE_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

// [MoE 模型原理 §4.1] C = ceil(c·T·k/E) for the exact binary value of c:
// write c = m·2^p with m a 53-bit integer; then C = ceil(m·T·k·2^p / E),
// evaluated in unsigned 128-bit integers.
static int64_t capacity_of(int64_t T, int32_t k, int32_t E, double c) {
  if (!(c >= std::ldexp(1.0, -30) && c <= std::ldexp(1.0, 30))) return -1;
  int p = 0;
  const double frac = std::frexp(c, &p);                 // c = frac·2^p, frac in [0.5, 1)
  unsigned long long m = (unsigned long long)std::ldexp(frac, 53);
  p -= 53;                                               // c = m·2^p
  const int tz = __builtin_ctzll(m);
  m >>= tz;
  p += tz;
  unsigned __int128 num = (unsigned __int128)m * (unsigned long long)T * (unsigned long long)k;
  unsigned __int128 den = (unsigned long long)E;
  if (p > 0) num <<= p;
  if (p < 0) den <<= -p;
  return (int64_t)(num / den + (num % den != 0 ? 1 : 0));
}

static moe_status_t check_cfg(const moe_config_t* c) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cfg is NULL");
  if (c->T < 1) return fail(MOE_ERR_INVALID_ARG, "T must be >= 1");
  if (c->E < 1 || c->E > 1024) return fail(MOE_ERR_INVALID_ARG, "E must be in [1, 1024]");
  if (c->k < 1 || c->k > 16 || c->k > c->E)
    return fail(MOE_ERR_INVALID_ARG, "k must be in [1, min(16, E)]");
  if (c->T * int64_t(c->k) >= (int64_t(1) << 31))
    return fail(MOE_ERR_INVALID_ARG, "T*k must be < 2^31");
  if (c->d < 8 || c->d % 8 != 0) return fail(MOE_ERR_INVALID_ARG, "d must be a multiple of 8");
  if (c->d_ff < 8 || c->d_ff % 8 != 0)
    return fail(MOE_ERR_INVALID_ARG, "d_ff must be a multiple of 8");
  if (!(c->capacity_factor >= std::ldexp(1.0, -30) && c->capacity_factor <= std::ldexp(1.0, 30)))
    return fail(MOE_ERR_INVALID_ARG, "capacity_factor must be in [2^-30, 2^30]");
  if (c->dtype != MOE_DT_F32 && c->dtype != MOE_DT_BF16)
    return fail(MOE_ERR_UNSUPPORTED, "dtype must be MOE_DT_F32 or MOE_DT_BF16");
  if (c->act != MOE_ACT_RELU && c->act != MOE_ACT_GELU_TANH)
    return fail(MOE_ERR_UNSUPPORTED, "act must be MOE_ACT_RELU or MOE_ACT_GELU_TANH");
  if (c->reroute != 0 && c->reroute != 1) return fail(MOE_ERR_INVALID_ARG, "reroute must be 0 or 1");
  if (c->fuse_dispatch != 0 && c->fuse_dispatch != 1)
    return fail(MOE_ERR_INVALID_ARG, "fuse_dispatch must be 0 or 1");
  if (c->fuse_combine != 0 && c->fuse_combine != 1)
    return fail(MOE_ERR_INVALID_ARG, "fuse_combine must be 0 or 1");
  return MOE_OK;
}

static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Arrival counters of the combine folded into the second GEMM: one per token,
// column tile and column half of that GEMM (N = d).
static size_t combine_counters(const moe_config_t& c) {
  const int bn = gemm_tc_bn(c.d);
  return size_t(c.T) * 2 * size_t((c.d + bn - 1) / bn);
}

static WsLayout layout_of(const moe_config_t& c) {
  WsLayout L{};
  L.n_chunks = (c.T + kChunkTokens - 1) / kChunkTokens;
  L.n_route_blocks = (c.T + kRouteTokensSimt - 1) / kRouteTokensSimt;
  size_t off = 0;
  L.status = off;
  off += kWsHeaderBytes;
  L.chunk_counts = off;
  off += align256(size_t(L.n_chunks) * c.E * sizeof(int32_t));
  L.psum_partial = off;
  off += align256(size_t(L.n_route_blocks) * c.E * sizeof(float));
  L.route_part = off;
  if (route_tc_supported(c))
    off += align256(size_t(route_tc_nsplit(c)) * size_t(c.T) * c.E * sizeof(float));
  L.reroute = off;
  if (c.reroute)
    off += 4 * align256(size_t(c.T) * c.k * sizeof(int32_t)) + 2 * align256(size_t(c.E) * 4);
  L.combine_cnt = off;
  if (c.fuse_combine) off += align256(combine_counters(c) * sizeof(int32_t));
  L.total = off;
  return L;
}

struct Ws {
  int32_t* status;
  int* route_counter;     // grid-completion counters (inside the status block)
  int* dispatch_counter;
  int* dispatch_barrier;  // int [2] for the one-pass dispatch's grid barrier
  int32_t* chunk_counts;
  float* psum_partial;
  float* route_part;
  unsigned long long* psum_fixed;
  RerouteBufs rr;  // all NULL unless cfg.reroute
  int32_t* cand;   // = rr.cand (written by the router)
  int* combine_cnt;  // NULL unless cfg.fuse_combine
};

static moe_status_t get_ws(const moe_config_t& c, void* ws, size_t ws_bytes, Ws* out) {
  const WsLayout L = layout_of(c);
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0)
    return fail(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (ws_bytes < L.total)
    return fail(MOE_ERR_WORKSPACE, "workspace smaller than moe_workspace_size()");
  char* b = static_cast<char*>(ws);
  out->status = reinterpret_cast<int32_t*>(b + L.status);
  out->route_counter = reinterpret_cast<int*>(b + L.status + kWsRouteCounter);
  out->dispatch_counter = reinterpret_cast<int*>(b + L.status + kWsDispatchCounter);
  out->dispatch_barrier = reinterpret_cast<int*>(b + L.status + kWsDispatchBarrier);
  out->chunk_counts = reinterpret_cast<int32_t*>(b + L.chunk_counts);
  out->psum_partial = reinterpret_cast<float*>(b + L.psum_partial);
  out->route_part = reinterpret_cast<float*>(b + L.route_part);
  out->psum_fixed = reinterpret_cast<unsigned long long*>(b + L.status + kWsPsumFixed);
  out->rr = RerouteBufs{};
  out->cand = nullptr;
  out->combine_cnt = c.fuse_combine ? reinterpret_cast<int*>(b + L.combine_cnt) : nullptr;
  if (c.reroute) {
    const size_t tk = align256(size_t(c.T) * c.k * sizeof(int32_t));
    char* r = b + L.reroute;
    out->cand = reinterpret_cast<int32_t*>(r);
    out->rr.cand = out->cand;
    out->rr.ids1 = reinterpret_cast<int32_t*>(r + tk);
    out->rr.pos0 = reinterpret_cast<int32_t*>(r + 2 * tk);
    out->rr.pos1 = reinterpret_cast<int32_t*>(r + 3 * tk);
    out->rr.kept0 = reinterpret_cast<int32_t*>(r + 4 * tk);
    out->rr.counts1 = reinterpret_cast<int32_t*>(r + 4 * tk + align256(size_t(c.E) * 4));
  }
  return MOE_OK;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Most rows any expert can hold: min(C, T·k) (kept = min(count, C)).
static int64_t rows_per_expert_max(const moe_config_t* c) {
  const int64_t C = capacity_of(c->T, c->k, c->E, c->capacity_factor);
  const int64_t tk = c->T * c->k;
  return C < tk ? C : tk;
}

// Which expert GEMM runs for bf16 layers: the tcgen05 kernel by default;
// MOE_FFN_IMPL=simt selects the CUDA-core kernel (a cross-check in tests).
static bool use_tc_gemm(const moe_config_t& c) {
  if (c.dtype != MOE_DT_BF16) return false;
  const char* v = std::getenv("MOE_FFN_IMPL");
  return !(v && std::strcmp(v, "simt") == 0);
}

// The gathering first GEMM and the combining second GEMM exist for the
// regular tcgen05 kernel only (bf16, more than 64 rows per expert possible).
static bool gather_supported(const moe_config_t& c) {
  return use_tc_gemm(c) && !gemm_swap_applies(rows_per_expert_max(&c));
}

// Which router runs.  bf16 layers: the tcgen05 router for E <= 256, else the
// generic CUDA-core router; fp32 layers: the generic CUDA-core router (tf32
// tensor cores would not meet an fp32 tolerance).  MOE_ROUTE_IMPL=simt|warp|tc
// forces one where it applies (the warp router, bf16 with E <= 32, is a
// cross-check: it measured slower than the tcgen05 router on these shapes).  Inputs that are not 16-byte aligned take the generic router.
enum class Router { kSimt, kWarp, kTc };
static Router pick_router(const moe_config_t& c, bool aligned) {
  // The warp and tcgen05 routers read x and W_r in 16-byte units.
  if (!aligned) return Router::kSimt;
  const char* v = std::getenv("MOE_ROUTE_IMPL");
  if (v && std::strcmp(v, "simt") == 0) return Router::kSimt;
  if (v && std::strcmp(v, "tc") == 0 && route_tc_supported(c)) return Router::kTc;
  if (v && std::strcmp(v, "warp") == 0 && route_warp_supported(c)) return Router::kWarp;
  if (route_tc_supported(c)) return Router::kTc;
  return Router::kSimt;
}

}  // namespace moe

namespace moe {
// moe_route.  psum_fixed_out == NULL: psum is written before return (every
// router).  Otherwise the tensor-core and CUDA-core routers leave Σ_t p in the
// workspace's fixed-point accumulators and set *psum_fixed_out to them, for
// the dispatch's histogram to convert (psum_from_fixed); the warp router
// writes psum and sets it to NULL.
static moe_status_t route_impl(const moe_config_t* cfg, const void* x, const void* Wr,
                               const float* br, const float* sel_bias, float* logits,
                               int32_t* topk_ids, float* topk_w, float* psum, void* ws,
                               size_t ws_bytes, unsigned long long** psum_fixed_out,
                               void* stream) {
  const StageRange range("moe_route");
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!x || !Wr || !br || !topk_ids || !topk_w || !psum)
    return fail(MOE_ERR_INVALID_ARG, "moe_route: NULL tensor");
  if (cfg->write_logits && !logits)
    return fail(MOE_ERR_INVALID_ARG, "moe_route: write_logits set but logits is NULL");
  Ws w;
  if ((s = get_ws(*cfg, ws, ws_bytes, &w)) != MOE_OK) return s;
  float* lg = cfg->write_logits ? logits : nullptr;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* counter = w.route_counter;
  if (psum_fixed_out) *psum_fixed_out = nullptr;
  cudaError_t e;
  switch (pick_router(*cfg, aligned16(x) && aligned16(Wr))) {
    case Router::kWarp:
      e = launch_route_warp(*cfg, x, Wr, br, lg, topk_ids, topk_w, w.psum_partial, psum, counter,
                            sel_bias, w.cand, st);
      break;
    case Router::kTc:
      e = launch_route_tc(*cfg, x, Wr, w.route_part, w.status, st);
      if (e == cudaSuccess)
        e = launch_route_select(*cfg, w.route_part, route_tc_nsplit(*cfg), br, lg, topk_ids,
                                topk_w, w.psum_fixed, psum, counter, psum_fixed_out == nullptr,
                                sel_bias, w.cand, st);
      if (e == cudaSuccess && psum_fixed_out) *psum_fixed_out = w.psum_fixed;
      break;
    default:
      e = launch_route_simt(*cfg, x, Wr, br, lg, topk_ids, topk_w, w.psum_fixed, psum, counter,
                            psum_fixed_out == nullptr, sel_bias, w.cand, st);
      if (e == cudaSuccess && psum_fixed_out) *psum_fixed_out = w.psum_fixed;
      break;
  }
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_route");
}
}  // namespace moe

using namespace moe;

extern "C" {

int64_t moe_capacity(const moe_config_t* cfg) {
  if (check_cfg(cfg) != MOE_OK) return -1;
  return capacity_of(cfg->T, cfg->k, cfg->E, cfg->capacity_factor);
}

int64_t moe_max_rows(const moe_config_t* cfg) {
  const int64_t C = moe_capacity(cfg);
  if (C < 0) return -1;
  const int64_t a = cfg->T * cfg->k, b = C * cfg->E;
  return a < b ? a : b;
}

moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!bytes) return fail(MOE_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = layout_of(*cfg).total;
  return MOE_OK;
}

moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < kWsHeaderBytes) return fail(MOE_ERR_INVALID_ARG, "workspace too small");
  cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_workspace_init");
}

moe_status_t moe_route(const moe_config_t* cfg, const void* x, const void* Wr, const float* br,
                       float* logits, int32_t* topk_ids, float* topk_w, float* psum, void* ws,
                       size_t ws_bytes, void* stream) {
  return route_impl(cfg, x, Wr, br, nullptr, logits, topk_ids, topk_w, psum, ws, ws_bytes,
                    nullptr, stream);
}

moe_status_t moe_route_sel(const moe_config_t* cfg, const void* x, const void* Wr,
                           const float* br, const float* sel_bias, float* logits,
                           int32_t* topk_ids, float* topk_w, float* psum, void* ws,
                           size_t ws_bytes, void* stream) {
  return route_impl(cfg, x, Wr, br, sel_bias, logits, topk_ids, topk_w, psum, ws, ws_bytes,
                    nullptr, stream);
}

moe_status_t moe_routing_health(const moe_config_t* cfg, const int32_t* counts,
                                const int32_t* kept, float* health, void* stream) {
  const StageRange range("moe_routing_health");
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!counts || !kept || !health)
    return fail(MOE_ERR_INVALID_ARG, "moe_routing_health: NULL tensor");
  cudaError_t e = launch_health(*cfg, counts, kept, health, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_routing_health");
}

}  // extern "C"

namespace moe {
// moe_dispatch, optionally with the f / p̄ / L_aux statistics computed by the
// histogram's last block (aux != NULL, as in moe_forward).
static moe_status_t dispatch_impl(const moe_config_t* cfg, const void* x,
                                  const int32_t* topk_ids, int32_t* counts, int32_t* kept,
                                  int32_t* offsets, int32_t* slot_row, int32_t* row_token,
                                  void* xd, void* ws, size_t ws_bytes, const AuxArgs* aux,
                                  void* stream) {
  const StageRange range("moe_dispatch");
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!x || !topk_ids || !counts || !kept || !offsets || !slot_row || !row_token ||
      (!xd && !cfg->fuse_dispatch))
    return fail(MOE_ERR_INVALID_ARG, "moe_dispatch: NULL tensor");
  // With fuse_dispatch the rows are not copied (xd may be NULL, and is not
  // written).
  if (cfg->fuse_dispatch) xd = nullptr;
  if (!aligned16(x) || (xd && !aligned16(xd)))
    return fail(MOE_ERR_INVALID_ARG, "moe_dispatch: x and xd must be 16-byte aligned");
  Ws w;
  if ((s = get_ws(*cfg, ws, ws_bytes, &w)) != MOE_OK) return s;
  const int64_t C = capacity_of(cfg->T, cfg->k, cfg->E, cfg->capacity_factor);
  cudaError_t e = launch_dispatch(*cfg, C, x, topk_ids, counts, kept, offsets, slot_row,
                                  row_token, xd, w.chunk_counts, w.status, w.dispatch_counter,
                                  w.dispatch_barrier, aux, cfg->reroute ? &w.rr : nullptr,
                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_dispatch");
}
}  // namespace moe

extern "C" {

moe_status_t moe_dispatch(const moe_config_t* cfg, const void* x, const int32_t* topk_ids,
                          int32_t* counts, int32_t* kept, int32_t* offsets, int32_t* slot_row,
                          int32_t* row_token, void* xd, void* ws, size_t ws_bytes, void* stream) {
  return dispatch_impl(cfg, x, topk_ids, counts, kept, offsets, slot_row, row_token, xd, ws,
                       ws_bytes, nullptr, stream);
}

moe_status_t moe_ffn_up(const moe_config_t* cfg, const void* xd, const int32_t* offsets,
                        const void* W1, const float* b1, void* H, void* ws, size_t ws_bytes,
                        void* stream) {
  const StageRange range("moe_ffn_up");
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!xd || !offsets || !W1 || !b1 || !H)
    return fail(MOE_ERR_INVALID_ARG, "moe_ffn_up: NULL tensor");
  if (!aligned16(xd) || !aligned16(W1) || !aligned16(H))
    return fail(MOE_ERR_INVALID_ARG, "moe_ffn_up: xd, W1, H must be 16-byte aligned");
  Ws w;
  if ((s = get_ws(*cfg, ws, ws_bytes, &w)) != MOE_OK) return s;
  const int64_t R = moe_max_rows(cfg);
  const int64_t rpe = rows_per_expert_max(cfg);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e =
      !use_tc_gemm(*cfg)
          ? launch_gemm_simt(cfg->dtype, cfg->E, cfg->d_ff, cfg->d, R, offsets, xd, W1, b1,
                             cfg->act, H, st)
      : gemm_swap_applies(rpe)
          ? launch_gemm_swap(cfg->E, cfg->d_ff, cfg->d, R, rpe, offsets, xd, W1, b1, cfg->act, H,
                             w.status, st)
          : launch_gemm_tc(cfg->E, cfg->d_ff, cfg->d, R, offsets, xd, W1, b1, cfg->act, H,
                           w.status, st);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_ffn_up");
}

moe_status_t moe_ffn_up_gather(const moe_config_t* cfg, const void* x, const int32_t* row_token,
                               const int32_t* offsets, const void* W1, const float* b1, void* H,
                               void* ws, size_t ws_bytes, void* stream) {
  const StageRange range("moe_ffn_up_gather");
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!x || !row_token || !offsets || !W1 || !b1 || !H)
    return fail(MOE_ERR_INVALID_ARG, "moe_ffn_up_gather: NULL tensor");
  if (!aligned16(x) || !aligned16(W1) || !aligned16(H))
    return fail(MOE_ERR_INVALID_ARG, "moe_ffn_up_gather: x, W1, H must be 16-byte aligned");
  if (!gather_supported(*cfg))
    return fail(MOE_ERR_UNSUPPORTED,
                "moe_ffn_up_gather: needs bf16 and the tensor-core GEMM for more than 64 rows "
                "per expert");
  Ws w;
  if ((s = get_ws(*cfg, ws, ws_bytes, &w)) != MOE_OK) return s;
  cudaError_t e = launch_gemm_tc_gather(cfg->E, cfg->d_ff, cfg->d, moe_max_rows(cfg), offsets, x,
                                        cfg->T, row_token, W1, b1, cfg->act, H, w.status,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_ffn_up_gather");
}

moe_status_t moe_ffn_down(const moe_config_t* cfg, const void* H, const int32_t* offsets,
                          const void* W2, const float* b2, void* yd, void* ws, size_t ws_bytes,
                          void* stream) {
  const StageRange range("moe_ffn_down");
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!H || !offsets || !W2 || !b2 || !yd)
    return fail(MOE_ERR_INVALID_ARG, "moe_ffn_down: NULL tensor");
  if (!aligned16(H) || !aligned16(W2) || !aligned16(yd))
    return fail(MOE_ERR_INVALID_ARG, "moe_ffn_down: H, W2, yd must be 16-byte aligned");
  Ws w;
  if ((s = get_ws(*cfg, ws, ws_bytes, &w)) != MOE_OK) return s;
  const int64_t R = moe_max_rows(cfg);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t rpe = rows_per_expert_max(cfg);
  cudaError_t e =
      !use_tc_gemm(*cfg)
          ? launch_gemm_simt(cfg->dtype, cfg->E, cfg->d, cfg->d_ff, R, offsets, H, W2, b2, -1,
                             yd, st)
      : gemm_swap_applies(rpe)
          ? launch_gemm_swap(cfg->E, cfg->d, cfg->d_ff, R, rpe, offsets, H, W2, b2, -1, yd,
                             w.status, st)
          : launch_gemm_tc(cfg->E, cfg->d, cfg->d_ff, R, offsets, H, W2, b2, -1, yd, w.status,
                           st);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_ffn_down");
}

moe_status_t moe_ffn_down_combine(const moe_config_t* cfg, const void* H, const int32_t* offsets,
                                  const int32_t* row_token, const int32_t* slot_row,
                                  const float* topk_w, const void* W2, const float* b2, void* yd,
                                  void* y, void* ws, size_t ws_bytes, void* stream) {
  const StageRange range("moe_ffn_down_combine");
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!H || !offsets || !row_token || !slot_row || !topk_w || !W2 || !b2 || !yd || !y)
    return fail(MOE_ERR_INVALID_ARG, "moe_ffn_down_combine: NULL tensor");
  if (!aligned16(H) || !aligned16(W2) || !aligned16(yd) || !aligned16(y))
    return fail(MOE_ERR_INVALID_ARG, "moe_ffn_down_combine: H, W2, yd, y must be 16-byte aligned");
  if (!cfg->fuse_combine)
    return fail(MOE_ERR_INVALID_ARG,
                "moe_ffn_down_combine: needs cfg->fuse_combine (its workspace holds the counters)");
  if (!gather_supported(*cfg))
    return fail(MOE_ERR_UNSUPPORTED,
                "moe_ffn_down_combine: needs bf16 and the tensor-core GEMM for more than 64 rows "
                "per expert");
  Ws w;
  if ((s = get_ws(*cfg, ws, ws_bytes, &w)) != MOE_OK) return s;
  cudaError_t e = launch_gemm_tc_combine(cfg->E, cfg->d, cfg->d_ff, moe_max_rows(cfg), offsets, H,
                                         W2, b2, yd, cfg->T, cfg->k, row_token, slot_row, topk_w,
                                         y, w.combine_cnt, w.status,
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_ffn_down_combine");
}

moe_status_t moe_expert_ffn(const moe_config_t* cfg, const void* xd, const int32_t* offsets,
                            const void* W1, const float* b1, const void* W2, const float* b2,
                            void* H, void* yd, void* ws, size_t ws_bytes, void* stream) {
  const StageRange range("moe_expert_ffn");
  moe_status_t s = moe_ffn_up(cfg, xd, offsets, W1, b1, H, ws, ws_bytes, stream);
  if (s != MOE_OK) return s;
  return moe_ffn_down(cfg, H, offsets, W2, b2, yd, ws, ws_bytes, stream);
}

moe_status_t moe_combine(const moe_config_t* cfg, const void* yd, const int32_t* slot_row,
                         const float* topk_w, void* y, void* stream) {
  const StageRange range("moe_combine");
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!yd || !slot_row || !topk_w || !y)
    return fail(MOE_ERR_INVALID_ARG, "moe_combine: NULL tensor");
  if (!aligned16(yd) || !aligned16(y))
    return fail(MOE_ERR_INVALID_ARG, "moe_combine: yd and y must be 16-byte aligned");
  cudaError_t e = launch_combine(*cfg, moe_max_rows(cfg), yd, slot_row, topk_w, y,
                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_combine");
}

moe_status_t moe_aux_stats(const moe_config_t* cfg, const int32_t* counts, const float* psum,
                           float alpha, float* f, float* pbar, float* l_aux, void* stream) {
  const StageRange range("moe_aux_stats");
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!counts || !psum || !f || !pbar || !l_aux)
    return fail(MOE_ERR_INVALID_ARG, "moe_aux_stats: NULL tensor");
  cudaError_t e = launch_aux(*cfg, counts, psum, alpha, f, pbar, l_aux,
                             static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_aux_stats");
}

moe_status_t moe_forward(const moe_config_t* cfg, const moe_tensors_t* t, float alpha, void* ws,
                         size_t ws_bytes, void* stream) {
  const StageRange range("moe_forward");
  if (!t) return fail(MOE_ERR_INVALID_ARG, "moe_forward: tensors is NULL");
  if (!t->f || !t->pbar || !t->l_aux)
    return fail(MOE_ERR_INVALID_ARG, "moe_aux_stats: NULL tensor");
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if ((cfg->fuse_dispatch || cfg->fuse_combine) && !gather_supported(*cfg))
    return fail(MOE_ERR_UNSUPPORTED,
                "moe_forward: fuse_dispatch and fuse_combine need bf16 and the tensor-core GEMM "
                "for more than 64 rows per expert");
  unsigned long long* psum_fixed = nullptr;
  if ((s = route_impl(cfg, t->x, t->Wr, t->br, t->sel_bias, t->logits, t->topk_ids, t->topk_w,
                      t->psum, ws, ws_bytes, &psum_fixed, stream)) != MOE_OK)
    return s;
  // The statistics need only counts and psum: the dispatch's last histogram
  // block computes them (same arithmetic as moe_aux_stats), saving a launch;
  // with the tensor-core router it first forms psum from the fixed-point sums.
  const AuxArgs aux{alpha, t->psum, t->f, t->pbar, t->l_aux, psum_fixed, t->health};
  if ((s = dispatch_impl(cfg, t->x, t->topk_ids, t->counts, t->kept, t->offsets, t->slot_row,
                         t->row_token, t->xd, ws, ws_bytes, &aux, stream)) != MOE_OK)
    return s;
  s = cfg->fuse_dispatch ? moe_ffn_up_gather(cfg, t->x, t->row_token, t->offsets, t->W1, t->b1,
                                              t->H, ws, ws_bytes, stream)
                         : moe_ffn_up(cfg, t->xd, t->offsets, t->W1, t->b1, t->H, ws, ws_bytes,
                                      stream);
  if (s != MOE_OK) return s;
  if (cfg->fuse_combine)
    return moe_ffn_down_combine(cfg, t->H, t->offsets, t->row_token, t->slot_row, t->topk_w,
                                t->W2, t->b2, t->yd, t->y, ws, ws_bytes, stream);
  if ((s = moe_ffn_down(cfg, t->H, t->offsets, t->W2, t->b2, t->yd, ws, ws_bytes, stream)) !=
      MOE_OK)
    return s;
  return moe_combine(cfg, t->yd, t->slot_row, t->topk_w, t->y, stream);
}

moe_status_t moe_selftest_wait_timeout(void* ws, size_t ws_bytes, int64_t limit_ns,
                                       void* stream) {
  if (!ws || ws_bytes < kWsHeaderBytes)
    return fail(MOE_ERR_INVALID_ARG, "moe_selftest_wait_timeout: workspace too small");
  if (limit_ns < 1000000 || limit_ns > 4000000000LL)
    return fail(MOE_ERR_INVALID_ARG, "moe_selftest_wait_timeout: limit_ns out of range");
  cudaError_t e = launch_wait_timeout_selftest(static_cast<int32_t*>(ws), uint64_t(limit_ns),
                                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_selftest_wait_timeout");
}

moe_status_t moe_selftest_grid_barrier_timeout(void* ws, size_t ws_bytes, int64_t limit_ns,
                                               void* stream) {
  if (!ws || ws_bytes < kWsHeaderBytes)
    return fail(MOE_ERR_INVALID_ARG, "moe_selftest_grid_barrier_timeout: workspace too small");
  if (limit_ns < 1000000 || limit_ns > 4000000000LL)
    return fail(MOE_ERR_INVALID_ARG, "moe_selftest_grid_barrier_timeout: limit_ns out of range");
  uint8_t* b = static_cast<uint8_t*>(ws);
  cudaError_t e = launch_grid_barrier_timeout_selftest(
      reinterpret_cast<int*>(b + kWsDispatchBarrier), reinterpret_cast<int32_t*>(b),
      uint64_t(limit_ns), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_selftest_grid_barrier_timeout");
}

moe_status_t moe_get_device_status(const void* ws, int32_t* status) {
  if (!ws || !status) return fail(MOE_ERR_INVALID_ARG, "moe_get_device_status: NULL argument");
  cudaError_t e = cudaMemcpy(status, ws, sizeof(int32_t), cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_get_device_status");
}

int64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    default: return "MOE_ERR_UNKNOWN";
  }
}

const char* moe_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
