// Plain CPU oracle for the forward pass of one Mixture-of-Experts layer.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
// calls this file; only the test suite, the smoke check and the benchmark's
// CPU-baseline leg do.  It shares no code, header, table or helper with the
// CUDA path.
//
// Every step is written out in the order the source article gives it, with
// plain loops and double accumulation, so that it can be checked by eye
// against the formulas.  The article is
//   "MoE 模型原理：路由、专家负载、容量、通信与推理成本" (wrblog.cn),
// cited below by section number, e.g. [MoE 模型原理 §4.1].  The capacity
// example with 1024 tokens comes from
//   "Expert Parallelism：为什么让 Token 去找 Expert，而不是搬运参数？"
// (111qqz.com), section "Expert Capacity 和 Token Dropping".
//
// Precision: bf16 values are stored as uint16 bit patterns and widened
// exactly to double by a 16-bit shift; every sum is accumulated in double.
// Parallelism: independent tokens (or buffer rows) are split across
// std::thread workers; each output element is still produced by one plain
// sequential loop, so the thread count never changes a result.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

namespace {

// Element readers: x, W_r, W1, W2 are either fp32 or bf16 (uint16 bits).
inline double bf16_bits_to_double(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

inline double load_elem(const void* base, int is_bf16, int64_t i) {
  if (is_bf16) return bf16_bits_to_double(static_cast<const uint16_t*>(base)[i]);
  return static_cast<double>(static_cast<const float*>(base)[i]);
}

// Round a double to the nearest bf16 (round-half-to-even), returned as double.
// Used only when the caller asks the oracle to mirror a bf16 intermediate.
inline double round_to_bf16(double v) {
  float f = static_cast<float>(v);
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u) return static_cast<double>(f);  // inf/nan
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  u &= 0xffff0000u;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

int worker_count(int64_t n_items) {
  unsigned hc = std::thread::hardware_concurrency();
  int64_t w = hc == 0 ? 1 : static_cast<int64_t>(hc);
  if (w > n_items) w = n_items;
  return w < 1 ? 1 : static_cast<int>(w);
}

// Run body(i) for i in [0, n) on a few threads, contiguous ranges each.
void parallel_for(int64_t n, const std::function<void(int64_t)>& body) {
  int nw = worker_count(n);
  if (nw <= 1) {
    for (int64_t i = 0; i < n; ++i) body(i);
    return;
  }
  std::vector<std::thread> pool;
  int64_t per = (n + nw - 1) / nw;
  for (int w = 0; w < nw; ++w) {
    int64_t lo = w * per, hi = std::min<int64_t>(n, lo + per);
    if (lo >= hi) break;
    pool.emplace_back([lo, hi, &body] {
      for (int64_t i = lo; i < hi; ++i) body(i);
    });
  }
  for (auto& t : pool) t.join();
}

// Expert activation σ.  [MoE 模型原理 §1] writes FFN(x)=W2 σ(W1 x+b1)+b2 and
// leaves σ open; the workloads use ReLU or the tanh form of GELU,
// 0.5·u·(1+tanh(√(2/π)·(u+0.044715·u³))).
double activation(int act, double u) {
  if (act == 0) return u > 0.0 ? u : 0.0;
  const double kPi = 3.14159265358979323846;
  double inner = std::sqrt(2.0 / kPi) * (u + 0.044715 * u * u * u);
  return 0.5 * u * (1.0 + std::tanh(inner));
}

}  // namespace

extern "C" {

int oracle_num_threads(void) { return worker_count(1 << 30); }

// [MoE 模型原理 §4.1]  C = ceil(c · T·k / E), evaluated exactly for the
// binary value of the double c: c = M·2^q with M an integer, so C is the
// ceiling of the rational M·T·k·2^q / E, done in 128-bit integers.
// Requires 2^-30 <= c <= 2^30 (returns -1 otherwise).
int64_t oracle_capacity(int64_t T, int32_t k, int32_t E, double c) {
  if (!(c >= std::ldexp(1.0, -30) && c <= std::ldexp(1.0, 30)) || T < 0 || k < 1 || E < 1)
    return -1;
  int q = 0;
  double m = std::frexp(c, &q);  // c = m·2^q, 0.5 <= m < 1
  uint64_t M = static_cast<uint64_t>(std::ldexp(m, 53));
  int sh = q - 53;  // c = M·2^sh exactly
  while (M != 0 && (M & 1u) == 0) {
    M >>= 1;
    ++sh;
  }
  unsigned __int128 num = static_cast<unsigned __int128>(M) * static_cast<uint64_t>(T) *
                          static_cast<uint64_t>(k);
  unsigned __int128 den = static_cast<unsigned __int128>(static_cast<uint64_t>(E));
  if (sh >= 0)
    num <<= sh;
  else
    den <<= -sh;
  return static_cast<int64_t>((num + den - 1) / den);
}

void oracle_activation(int64_t n, int32_t act, const double* u, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = activation(act, u[i]);
}

// [MoE 模型原理 §2.1]  s_t = W_r x_t + b_r,  W_r ∈ R^{E×d} (row i = expert i).
// Output: logits[t*E + i] in double.
void oracle_router_logits(int64_t T, int32_t d, int32_t E, const void* x, int32_t x_bf16,
                          const void* Wr, int32_t w_bf16, const float* br, double* logits) {
  parallel_for(T, [&](int64_t t) {
    for (int32_t i = 0; i < E; ++i) {
      double s = 0.0;
      for (int32_t j = 0; j < d; ++j)
        s += load_elem(Wr, w_bf16, static_cast<int64_t>(i) * d + j) *
             load_elem(x, x_bf16, t * d + j);
      logits[t * E + i] = s + (br ? static_cast<double>(br[i]) : 0.0);
    }
  });
}

// [MoE 模型原理 §2.1, §2.2]  From fp32 logits s_t:
//   p_{t,i} = exp(s_{t,i}) / Σ_j exp(s_{t,j})      (evaluated as exp(s-max))
//   S_t     = TopK(p_t, k): the k largest, in descending order.  Softmax is
//             strictly increasing, so ranking s ranks p; ranking the fp32 s
//             avoids exp rounding creating or breaking ties.  Equal scores go
//             to the lower expert index (the article is silent on ties).
//   weights = p_{t,i} / Σ_{j∈S_t} p_{t,j}  if renormalize, else p_{t,i}
//             (§2.2 notes that some implementations do not renormalise).
// psum[i] = Σ_t p_{t,i}, summed over t in ascending order (for p̄, §3.2).
// sel_bias (nullable, [E]): a per-expert bias that moves only the choice of
// S_t (the expert-bias routing of [EP 工程 ai-master, 一、负载均衡]: it replaces the
// auxiliary loss and shifts which experts win, not the combine weights):
// experts are ranked by key_i = s_{t,i} + sel_bias_i, formed in fp32 (a
// float addition, the precision the selection is taken in), and the weights
// above still use the unbiased p.
// cand (nullable, [T,k]): the experts ranked k .. 2k-1 by the same keys (the
// next candidates of the ranked list, [MoE 模型原理 §4.3]), -1 past E.
void oracle_select(int64_t T, int32_t E, int32_t k, int32_t renormalize, const float* logits,
                   const float* sel_bias, int32_t* topk_ids, double* topk_w,
                   double* probs /*nullable, [T,E]*/, double* psum, int32_t* cand) {
  std::vector<double> p_all(static_cast<size_t>(T) * E);
  parallel_for(T, [&](int64_t t) {
    const float* s = logits + t * E;
    double mx = -INFINITY;
    for (int32_t i = 0; i < E; ++i) mx = std::max(mx, static_cast<double>(s[i]));
    double z = 0.0;
    for (int32_t i = 0; i < E; ++i) z += std::exp(static_cast<double>(s[i]) - mx);
    double* p = &p_all[static_cast<size_t>(t) * E];
    for (int32_t i = 0; i < E; ++i) p[i] = std::exp(static_cast<double>(s[i]) - mx) / z;

    // Ranking keys: the scores, or the scores plus the selection bias.
    std::vector<float> key(s, s + E);
    if (sel_bias)
      for (int32_t i = 0; i < E; ++i) key[i] = s[i] + sel_bias[i];
    // Top-k by repeated selection of the maximum among the not-yet-taken
    // experts; a strict '>' keeps the lowest index among equal keys.
    std::vector<char> taken(E, 0);
    double sel_sum = 0.0;
    for (int32_t r = 0; r < k; ++r) {
      int32_t best = -1;
      for (int32_t i = 0; i < E; ++i) {
        if (taken[i]) continue;
        if (best < 0 || key[i] > key[best]) best = i;
      }
      taken[best] = 1;
      topk_ids[t * k + r] = best;
      sel_sum += p[best];
    }
    for (int32_t r = 0; r < k; ++r) {
      double pr = p[topk_ids[t * k + r]];
      topk_w[t * k + r] = renormalize ? pr / sel_sum : pr;
    }
    if (cand) {
      // Continue the same selection for ranks k .. 2k-1.
      for (int32_t r = 0; r < k; ++r) {
        int32_t best = -1;
        for (int32_t i = 0; i < E; ++i) {
          if (taken[i]) continue;
          if (best < 0 || key[i] > key[best]) best = i;
        }
        cand[t * k + r] = best;
        if (best >= 0) taken[best] = 1;
      }
    }
  });
  for (int32_t i = 0; i < E; ++i) psum[i] = 0.0;
  for (int64_t t = 0; t < T; ++t)
    for (int32_t i = 0; i < E; ++i) psum[i] += p_all[static_cast<size_t>(t) * E + i];
  if (probs) std::memcpy(probs, p_all.data(), sizeof(double) * p_all.size());
}

// [MoE 模型原理 §4.2, §4.3]  Capacity assignment, first come first served.
// Slots are visited in (token, rank) order; slot (t,r) takes the next free
// position of its expert e; it is kept iff that position is below C.  Overflow
// is dropped (the first policy of §4.3) and capacity never moves between
// experts (§4.2).  Then the kept slots are laid out expert by expert:
//   kept[e]    = min(counts[e], C)
//   offsets[e] = Σ_{e'<e} kept[e']          (offsets[E] = total kept rows)
//   slot_row[t*k+r] = offsets[e] + position, or -1 when dropped
//   row_token[row]  = t
// counts[e] is the number of slots routed to e before capacity.
void oracle_fill(int64_t T, int32_t E, int32_t k, int64_t C, const int32_t* topk_ids,
                 int32_t* counts, int32_t* kept, int32_t* offsets, int32_t* slot_row,
                 int32_t* row_token) {
  std::vector<int64_t> position(static_cast<size_t>(T) * k);
  std::vector<int64_t> fill(E, 0);
  for (int64_t t = 0; t < T; ++t)
    for (int32_t r = 0; r < k; ++r) {
      int32_t e = topk_ids[t * k + r];
      position[t * k + r] = fill[e]++;
    }
  for (int32_t e = 0; e < E; ++e) {
    counts[e] = static_cast<int32_t>(fill[e]);
    kept[e] = static_cast<int32_t>(std::min<int64_t>(fill[e], C));
  }
  offsets[0] = 0;
  for (int32_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + kept[e];
  for (int64_t t = 0; t < T; ++t)
    for (int32_t r = 0; r < k; ++r) {
      int32_t e = topk_ids[t * k + r];
      int64_t pos = position[t * k + r];
      if (pos < C) {
        int32_t row = offsets[e] + static_cast<int32_t>(pos);
        slot_row[t * k + r] = row;
        row_token[row] = static_cast<int32_t>(t);
      } else {
        slot_row[t * k + r] = -1;
      }
    }
}

// [MoE 模型原理 §4.3], second policy: an overflowing slot goes to the next
// expert of the token's candidate list.  The page leaves open whether capacity
// is cut after the first assignment or assigned candidate by candidate; this
// takes the first assignment as oracle_fill does, then offers the overflow:
//   1. first-come fill in (token, rank) order: kept0[e] = min(counts[e], C);
//   2. the m-th overflowing slot of token t (in rank order) is offered to the
//      token's next candidate cand[t*k + m] (its expert of rank k + m); no
//      candidate (-1): the slot stays dropped;
//   3. offers are served first come in (token, rank) order of the offering
//      slot, into the room C - kept0[e] left after step 1; the rest drop.
// Buffer layout: an expert's first-fill rows, then its rerouted rows;
// kept[e] = kept0[e] + served[e], offsets = exclusive scan of kept.  counts
// stay those of the first choices (f_i is defined over S_t, §3.2); a
// rerouted slot keeps its combine weight (the caller's topk_w).
void oracle_fill_reroute(int64_t T, int32_t E, int32_t k, int64_t C, const int32_t* topk_ids,
                         const int32_t* cand, int32_t* counts, int32_t* kept, int32_t* offsets,
                         int32_t* slot_row, int32_t* row_token, int32_t* slot_expert) {
  const int64_t n = T * k;
  std::vector<int64_t> pos0(n), pos1(n, -1);
  std::vector<int32_t> dest(n, -1);
  std::vector<int64_t> fill(E, 0), served(E, 0), kept0(E);
  for (int64_t s = 0; s < n; ++s) pos0[s] = fill[topk_ids[s]]++;
  for (int32_t e = 0; e < E; ++e) {
    counts[e] = static_cast<int32_t>(fill[e]);
    kept0[e] = std::min<int64_t>(fill[e], C);
  }
  for (int64_t t = 0; t < T; ++t) {
    int32_t m = 0;
    for (int32_t r = 0; r < k; ++r) {
      const int64_t s = t * k + r;
      if (pos0[s] < C) {
        dest[s] = topk_ids[s];
        continue;
      }
      const int32_t e2 = m < k ? cand[t * k + m] : -1;
      ++m;
      if (e2 < 0) continue;
      if (served[e2] < C - kept0[e2]) {
        pos1[s] = served[e2]++;
        dest[s] = e2;
      }
    }
  }
  offsets[0] = 0;
  for (int32_t e = 0; e < E; ++e) {
    kept[e] = static_cast<int32_t>(kept0[e] + served[e]);
    offsets[e + 1] = offsets[e] + kept[e];
  }
  for (int64_t s = 0; s < n; ++s) {
    int32_t row = -1;
    if (dest[s] >= 0) {
      const int32_t e = dest[s];
      row = offsets[e] + static_cast<int32_t>(pos0[s] < C && dest[s] == topk_ids[s]
                                                  ? pos0[s]
                                                  : kept0[e] + pos1[s]);
      row_token[row] = static_cast<int32_t>(s / k);
    }
    slot_row[s] = row;
    if (slot_expert) slot_expert[s] = dest[s];
  }
}

// [MoE 模型原理 §5]  Dispatch: gather token rows into the per-expert buffer,
// xd[row] = x[row_token[row]], an exact byte copy.
void oracle_permute(int64_t n_rows, int64_t row_bytes, const void* x, const int32_t* row_token,
                    void* xd) {
  const char* src = static_cast<const char*>(x);
  char* dst = static_cast<char*>(xd);
  for (int64_t row = 0; row < n_rows; ++row)
    std::memcpy(dst + row * row_bytes, src + static_cast<int64_t>(row_token[row]) * row_bytes,
                static_cast<size_t>(row_bytes));
}

// [MoE 模型原理 §1]  Expert FFN on buffer rows:
//   h = σ(W1[e] x + b1[e]),  y = W2[e] h + b2[e],
// W1[e] ∈ R^{d_ff×d} (maps d → d_ff), W2[e] ∈ R^{d×d_ff} (maps d_ff → d).
// The expert owning a row is the e with offsets[e] <= row < offsets[e+1].
// Computes the n_sel rows listed in rows[] (all rows when rows == NULL,
// n_sel = offsets[E]); output yd_out[i*d + j] for the i-th listed row.
// round_h: 0 keeps h in double; 1 rounds h to bf16; 2 rounds h to fp32
// (mirrors a device that stores the hidden activation at that precision).
void oracle_ffn_rows(int32_t d, int32_t d_ff, int32_t E, const int32_t* offsets, int64_t n_sel,
                     const int32_t* rows, const void* xd, int32_t x_bf16, const void* W1,
                     const float* b1, const void* W2, const float* b2, int32_t w_bf16,
                     int32_t act, int32_t round_h, double* yd_out) {
  parallel_for(n_sel, [&](int64_t i) {
    int64_t row = rows ? rows[i] : i;
    int32_t e = 0;
    while (e < E && !(offsets[e] <= row && row < offsets[e + 1])) ++e;
    std::vector<double> h(d_ff);
    std::vector<double> xv(d);
    for (int32_t j = 0; j < d; ++j) xv[j] = load_elem(xd, x_bf16, row * d + j);
    const int64_t w1_base = static_cast<int64_t>(e) * d_ff * d;
    for (int32_t n = 0; n < d_ff; ++n) {
      double u = 0.0;
      for (int32_t j = 0; j < d; ++j) u += load_elem(W1, w_bf16, w1_base + int64_t(n) * d + j) * xv[j];
      u += b1 ? static_cast<double>(b1[int64_t(e) * d_ff + n]) : 0.0;
      double a = activation(act, u);
      if (round_h == 1) a = round_to_bf16(a);
      if (round_h == 2) a = static_cast<double>(static_cast<float>(a));
      h[n] = a;
    }
    const int64_t w2_base = static_cast<int64_t>(e) * d * d_ff;
    for (int32_t j = 0; j < d; ++j) {
      double y = 0.0;
      for (int32_t n = 0; n < d_ff; ++n) y += load_elem(W2, w_bf16, w2_base + int64_t(j) * d_ff + n) * h[n];
      y += b2 ? static_cast<double>(b2[int64_t(e) * d + j]) : 0.0;
      yd_out[i * d + j] = y;
    }
  });
}

// [MoE 模型原理 §2.2, §5]  Combine: y_t = Σ_{r : slot kept} w_{t,r} · yd[slot_row],
// summed in rank order r = 0..k-1.  A token whose every slot was dropped gets
// 0 (the residual add belongs to the caller).  Kept weights are not
// renormalised after a drop.
// Computes the n_sel tokens listed in tokens[] (all when tokens == NULL).
// yd rows are looked up through row_index[row] (an index into yd_rows), so a
// caller may pass only the rows that the selected tokens need.
void oracle_combine(int64_t n_sel, const int64_t* tokens, int32_t k, int32_t d,
                    const int32_t* slot_row, const double* topk_w, const int64_t* row_index,
                    const double* yd_rows, double* y_out) {
  parallel_for(n_sel, [&](int64_t i) {
    int64_t t = tokens ? tokens[i] : i;
    for (int32_t j = 0; j < d; ++j) y_out[i * d + j] = 0.0;
    for (int32_t r = 0; r < k; ++r) {
      int32_t row = slot_row[t * k + r];
      if (row < 0) continue;
      int64_t src = row_index ? row_index[row] : row;
      double w = topk_w[t * k + r];
      for (int32_t j = 0; j < d; ++j) y_out[i * d + j] += w * yd_rows[src * d + j];
    }
  });
}

// [MoE 模型原理 §3.2]  f_i = (1/T) Σ_t 1[i ∈ S_t] = counts_i / T (before
// capacity), p̄_i = (1/T) Σ_t p_{t,i}, L_aux = α · E · Σ_i f_i p̄_i.
void oracle_aux(int32_t E, int64_t T, double alpha, const int32_t* counts, const double* psum,
                double* f, double* pbar, double* l_aux) {
  double acc = 0.0;
  for (int32_t i = 0; i < E; ++i) {
    f[i] = static_cast<double>(counts[i]) / static_cast<double>(T);
    pbar[i] = psum[i] / static_cast<double>(T);
    acc += f[i] * pbar[i];
  }
  *l_aux = alpha * static_cast<double>(E) * acc;
}

// Routing-health indicators ([EP 工程 ai-master, 追问 2]: the entropy of the
// expert-activation distribution and the variance of the tokens each expert
// processes; [MoE 模型原理 §10.4]: the overflow share), from the counts
// before capacity and the kept rows after it:
//   out[0] = H = -Σ_i q_i ln q_i,  q_i = counts_i / (T·k)  (0·ln 0 = 0; nats)
//   out[1] = (1/E) Σ_i (counts_i - T·k/E)^2      (variance of routed slots)
//   out[2] = (1/E) Σ_i (kept_i - mean(kept))^2   (variance of processed rows)
//   out[3] = 1 - Σ_i kept_i / (T·k)              (fraction of slots dropped)
void oracle_routing_health(int32_t E, int64_t T, int32_t k, const int32_t* counts,
                           const int32_t* kept, double* out) {
  const double n = static_cast<double>(T) * static_cast<double>(k);
  double h = 0.0, vc = 0.0, vk = 0.0, kept_sum = 0.0;
  for (int32_t i = 0; i < E; ++i) {
    const double q = static_cast<double>(counts[i]) / n;
    if (q > 0.0) h -= q * std::log(q);
    kept_sum += static_cast<double>(kept[i]);
  }
  const double mc = n / static_cast<double>(E);
  const double mk = kept_sum / static_cast<double>(E);
  for (int32_t i = 0; i < E; ++i) {
    vc += (counts[i] - mc) * (counts[i] - mc);
    vk += (kept[i] - mk) * (kept[i] - mk);
  }
  out[0] = h;
  out[1] = vc / static_cast<double>(E);
  out[2] = vk / static_cast<double>(E);
  out[3] = 1.0 - kept_sum / n;
}

}  // extern "C"
