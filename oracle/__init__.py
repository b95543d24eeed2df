"""CPU oracle for the forward pass of one Mixture-of-Experts layer.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
library never links, loads or calls it, and it shares no code with the CUDA
path: the arithmetic lives in ``moe_oracle.cpp`` (plain loops, double
accumulation), and this module only marshals numpy arrays into it and chains
the steps in the order of the source article,

    "MoE 模型原理：路由、专家负载、容量、通信与推理成本" (wrblog.cn),

    §2.1 router scores and softmax  -> router_logits, select
    §2.2 top-k and renormalisation  -> select
    §4.1 capacity                   -> capacity
    §4.2/§4.3 first-come fill, drop -> fill
    §5   dispatch / combine         -> permute, combine
    §1   expert FFN                 -> ffn_rows
    §3.2 f_i, p̄_i, L_aux            -> aux

and, from "MoE Expert Parallelism 工程" (ai-master.cc), the expert-bias
selection (select's ``sel_bias``) and the routing-health indicators
(routing_health).

bf16 tensors are passed as numpy ``uint16`` arrays holding the bit patterns.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_lib = None
_lock = threading.Lock()

ACT_RELU = 0
ACT_GELU_TANH = 1


def build(force: bool = False) -> str:
    """Compile moe_oracle.cpp into libmoe_oracle.so beside it (g++, -O2)."""
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread",
                               _SRC, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.oracle_capacity.restype = i64
            lib.oracle_capacity.argtypes = [i64, i32, i32, f64]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_activation.argtypes = [i64, i32, P, P]
            lib.oracle_router_logits.argtypes = [i64, i32, i32, P, i32, P, i32, P, P]
            lib.oracle_select.argtypes = [i64, i32, i32, i32, P, P, P, P, P, P, P]
            lib.oracle_fill_reroute.argtypes = [i64, i32, i32, i64, P, P, P, P, P, P, P, P]
            lib.oracle_fill.argtypes = [i64, i32, i32, i64, P, P, P, P, P, P]
            lib.oracle_permute.argtypes = [i64, i64, P, P, P]
            lib.oracle_ffn_rows.argtypes = [i32, i32, i32, P, i64, P, P, i32, P, P, P, P, i32,
                                            i32, i32, P]
            lib.oracle_combine.argtypes = [i64, P, i32, i32, P, P, P, P, P]
            lib.oracle_aux.argtypes = [i32, i64, f64, P, P, P, P, P]
            lib.oracle_routing_health.argtypes = [i32, i64, i32, P, P, P]
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _elem(a):
    """Return (contiguous array, is_bf16) for an fp32 or bf16-bits array."""
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a), 1
    return _c(a, np.float32), 0


def num_threads() -> int:
    return int(_get().oracle_num_threads())


def capacity(T: int, k: int, E: int, c: float) -> int:
    """[§4.1] C = ceil(c·T·k/E)."""
    return int(_get().oracle_capacity(int(T), int(k), int(E), float(c)))


def activation(u, act: int):
    u = _c(u, np.float64)
    out = np.empty_like(u)
    _get().oracle_activation(u.size, int(act), _p(u), _p(out))
    return out


def router_logits(x, Wr, br):
    """[§2.1] s = W_r x + b_r in double; x [T,d], Wr [E,d] (fp32 or bf16 bits)."""
    x, xb = _elem(x)
    Wr, wb = _elem(Wr)
    T, d = x.shape
    E = Wr.shape[0]
    br = None if br is None else _c(br, np.float32)
    out = np.empty((T, E), np.float64)
    _get().oracle_router_logits(T, d, E, _p(x), xb, _p(Wr), wb, _p(br), _p(out))
    return out


def select(logits32, k: int, renormalize: bool, want_probs: bool = False, sel_bias=None,
           want_cand: bool = False):
    """[§2.1, §2.2] softmax, top-k (ties to the lower index), weights, Σ_t p.

    ``logits32`` are fp32 scores (the oracle's own, rounded, or a device's).
    ``sel_bias`` (fp32 [E] or None): experts are ranked by the fp32 sum
    score + sel_bias; the weights still come from the unbiased softmax.
    Returns (topk_ids int32 [T,k], topk_w float64 [T,k], psum float64 [E],
    probs float64 [T,E] or None), and with ``want_cand`` also cand int32
    [T,k]: the experts of rank k .. 2k-1 (-1 past E).
    """
    s = _c(logits32, np.float32)
    T, E = s.shape
    sb = None if sel_bias is None else _c(sel_bias, np.float32)
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    psum = np.empty(E, np.float64)
    probs = np.empty((T, E), np.float64) if want_probs else None
    cand = np.empty((T, k), np.int32) if want_cand else None
    _get().oracle_select(T, E, int(k), int(bool(renormalize)), _p(s), _p(sb), _p(ids), _p(w),
                         _p(probs), _p(psum), _p(cand))
    if want_cand:
        return ids, w, psum, probs, cand
    return ids, w, psum, probs


def fill(topk_ids, E: int, C: int):
    """[§4.2, §4.3] first-come capacity fill in (token, rank) order, drop overflow.

    Returns dict(counts, kept, offsets [E+1], slot_row [T,k], row_token [n_rows]).
    """
    ids = _c(topk_ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    kept = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    slot_row = np.empty((T, k), np.int32)
    row_token = np.full(max(T * k, 1), -1, np.int32)
    _get().oracle_fill(T, int(E), k, int(C), _p(ids), _p(counts), _p(kept), _p(offsets),
                       _p(slot_row), _p(row_token))
    n_rows = int(offsets[E])
    return dict(counts=counts, kept=kept, offsets=offsets, slot_row=slot_row,
                row_token=row_token[:n_rows].copy())


def permute(x, row_token):
    """[§5] xd[row] = x[row_token[row]] (exact copy)."""
    x = np.ascontiguousarray(x)
    rt = _c(row_token, np.int32)
    xd = np.empty((rt.shape[0],) + x.shape[1:], x.dtype)
    row_bytes = x.strides[0]
    _get().oracle_permute(rt.shape[0], row_bytes, _p(x), _p(rt), _p(xd))
    return xd


def ffn_rows(xd, offsets, W1, b1, W2, b2, act: int, rows=None, round_h: int = 0):
    """[§1] y = W2[e] σ(W1[e] x + b1[e]) + b2[e] for buffer rows (double out).

    xd [n_rows, d]; W1 [E, d_ff, d]; W2 [E, d, d_ff]; biases fp32.
    ``rows`` selects a subset of buffer rows (default: all offsets[E] rows).
    ``round_h``: 0 double, 1 bf16, 2 fp32 rounding of the hidden activation.
    """
    xd, xb = _elem(xd)
    W1, wb = _elem(W1)
    W2, wb2 = _elem(W2)
    assert wb == wb2
    E, d_ff, d = W1.shape
    offsets = _c(offsets, np.int32)
    if rows is None:
        rows_a = None
        n_sel = int(offsets[E])
    else:
        rows_a = _c(rows, np.int32)
        n_sel = rows_a.shape[0]
    b1 = None if b1 is None else _c(b1, np.float32)
    b2 = None if b2 is None else _c(b2, np.float32)
    out = np.empty((n_sel, d), np.float64)
    if n_sel:
        _get().oracle_ffn_rows(d, d_ff, E, _p(offsets), n_sel, _p(rows_a), _p(xd), xb, _p(W1),
                               _p(b1), _p(W2), _p(b2), wb, int(act), int(round_h), _p(out))
    return out


def combine(slot_row, topk_w, yd_rows, d: int, tokens=None, row_index=None):
    """[§2.2, §5] y_t = Σ_r w[t,r]·yd[slot_row[t,r]] over kept slots, rank order."""
    slot_row = _c(slot_row, np.int32)
    T, k = slot_row.shape
    w = _c(topk_w, np.float64)
    yd_rows = _c(yd_rows, np.float64)
    tok = None if tokens is None else _c(tokens, np.int64)
    n_sel = T if tok is None else tok.shape[0]
    ri = None if row_index is None else _c(row_index, np.int64)
    out = np.empty((n_sel, d), np.float64)
    if n_sel:
        _get().oracle_combine(n_sel, _p(tok), k, int(d), _p(slot_row), _p(w), _p(ri),
                              _p(yd_rows), _p(out))
    return out


def aux(counts, psum, T: int, alpha: float):
    """[§3.2] f = counts/T, p̄ = psum/T, L_aux = α·E·Σ f·p̄."""
    counts = _c(counts, np.int32)
    psum = _c(psum, np.float64)
    E = counts.shape[0]
    f = np.empty(E, np.float64)
    pbar = np.empty(E, np.float64)
    l = np.empty(1, np.float64)
    _get().oracle_aux(E, int(T), float(alpha), _p(counts), _p(psum), _p(f), _p(pbar), _p(l))
    return f, pbar, float(l[0])


def fill_reroute(topk_ids, cand, E: int, C: int):
    """[§4.3] first-come fill, then each overflowing slot offered once to its
    token's next candidate (see oracle_fill_reroute).  Returns fill()'s dict
    plus slot_expert [T,k] (the expert that processes each slot, -1 dropped).
    """
    ids = _c(topk_ids, np.int32)
    cd = _c(cand, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    kept = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    slot_row = np.empty((T, k), np.int32)
    slot_expert = np.empty((T, k), np.int32)
    row_token = np.full(max(T * k, 1), -1, np.int32)
    _get().oracle_fill_reroute(T, int(E), k, int(C), _p(ids), _p(cd), _p(counts), _p(kept),
                               _p(offsets), _p(slot_row), _p(row_token), _p(slot_expert))
    n_rows = int(offsets[E])
    return dict(counts=counts, kept=kept, offsets=offsets, slot_row=slot_row,
                row_token=row_token[:n_rows].copy(), slot_expert=slot_expert)


def routing_health(counts, kept, T: int, k: int):
    """Routing-health indicators from counts (before capacity) and kept rows:
    (entropy of counts/(T·k) in nats, variance of counts, variance of kept,
    fraction of slots dropped)."""
    counts = _c(counts, np.int32)
    kept = _c(kept, np.int32)
    out = np.empty(4, np.float64)
    _get().oracle_routing_health(counts.shape[0], int(T), int(k), _p(counts), _p(kept), _p(out))
    return out


def forward(x, Wr, br, W1, b1, W2, b2, *, k: int, capacity_factor: float, renormalize: bool,
            act: int, alpha: float = 1.0, logits32=None, tokens=None, round_h: int = 0,
            sel_bias=None, reroute: bool = False):
    """The whole layer, step by step in the article's order.

    ``logits32``: fp32 scores to route on (a device's own); default: the
    oracle's double scores rounded to fp32.  ``tokens``: compute the expert
    FFN and combine only for these tokens (routing always covers all T,
    because capacity positions depend on every earlier token).
    Returns a dict of every intermediate and output.
    """
    T = x.shape[0]
    E = Wr.shape[0]
    out = {}
    if logits32 is None:
        ld = router_logits(x, Wr, br)
        out["logits_f64"] = ld
        logits32 = ld.astype(np.float32)
    out["logits"] = np.asarray(logits32, np.float32)
    ids, w, psum, _, cand = select(logits32, k, renormalize, sel_bias=sel_bias, want_cand=True)
    out.update(topk_ids=ids, topk_w=w, psum=psum, cand=cand)
    C = capacity(T, k, E, capacity_factor)
    out["C"] = C
    fl = fill_reroute(ids, cand, E, C) if reroute else fill(ids, E, C)
    out.update(fl)
    f, pbar, l_aux = aux(fl["counts"], psum, T, alpha)
    out.update(f=f, pbar=pbar, l_aux=l_aux)
    out["health"] = routing_health(fl["counts"], fl["kept"], T, k)
    slot_row = fl["slot_row"]
    if tokens is None:
        xd = permute(x, fl["row_token"])
        out["xd"] = xd
        yd = ffn_rows(xd, fl["offsets"], W1, b1, W2, b2, act, round_h=round_h)
        out["yd"] = yd
        out["y"] = combine(slot_row, w, yd, x.shape[1])
    else:
        tokens = np.asarray(tokens, np.int64)
        rows = slot_row[tokens].reshape(-1)
        rows = np.unique(rows[rows >= 0]).astype(np.int32)
        row_index = np.full(int(fl["offsets"][E]) + 1, -1, np.int64)
        row_index[rows] = np.arange(rows.shape[0])
        # rows of the per-expert buffer hold token rows: xd[row] = x[row_token[row]]
        xd_sel = permute(x, fl["row_token"][rows]) if rows.size else x[:0]
        off_sel = _rows_offsets_for(rows, fl["offsets"])
        yd = ffn_rows(xd_sel, off_sel, W1, b1, W2, b2, act, round_h=round_h)
        out["rows"] = rows
        out["yd_rows"] = yd
        out["y"] = combine(slot_row, w, yd, x.shape[1], tokens=tokens, row_index=row_index)
    return out


def _rows_offsets_for(rows, offsets):
    """Expert boundaries of a sorted row subset, so ffn_rows finds each row's expert."""
    E = offsets.shape[0] - 1
    return np.searchsorted(rows, offsets[: E + 1], side="left").astype(np.int32)
