"""Helpers for the GPU-vs-oracle parity tests (imported by test files).

The CUDA path runs through the C ABI (routing_dispatch_expert_06_b300.moe);
the oracle runs on host copies of the same seeded tensors.  Tolerances:

* integer outputs (ids, counts, offsets, slot_row, row_token) and the
  permuted rows: bit-exact, with the oracle routing on the device's own fp32
  logits (so both sides take the top-k decision on the same numbers);
* logits: |a-b| <= 1e-5 · max(|b|, rms(row of b));
* other fp32 outputs: |a-b| <= 1e-4 · max(|b|, rms(row of b));
* bf16 outputs: |a-b| <= 1e-2 + 2e-2·|b|.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from routing_dispatch_expert_06_b300 import inputs, moe

ACT = {"relu": oracle.ACT_RELU, "gelu_tanh": oracle.ACT_GELU_TANH}


def h(t):
    return inputs.to_numpy(t)


def f64(t_or_a):
    a = h(t_or_a) if isinstance(t_or_a, torch.Tensor) else t_or_a
    return inputs.as_f64(a)


def assert_rel_rms(got, ref, rtol, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if ref.ndim == 1:
        scale = np.maximum(np.abs(ref), np.sqrt(np.mean(ref * ref)) if ref.size else 0.0)
    else:
        rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
        scale = np.maximum(np.abs(ref), rms)
    err = np.abs(got - ref)
    bad = err > rtol * scale + 1e-30
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} beyond rtol {rtol}; first at "
                             f"{tuple(i)}: got {got[tuple(i)]!r} ref {ref[tuple(i)]!r}")


def assert_bf16(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    bad = np.abs(got - ref) > 1e-2 + 2e-2 * np.abs(ref)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} beyond bf16 tolerance; first at "
                             f"{tuple(i)}: got {got[tuple(i)]!r} ref {ref[tuple(i)]!r}")


def assert_float(got, ref, dtype, what=""):
    if dtype == "bf16":
        assert_bf16(got, ref, what)
    else:
        assert_rel_rms(got, ref, 1e-4, what)


def run_gpu(wl, inp=None, expert_bias=False, alpha=1.0, stages=False, health=False,
            reroute=False, fuse_dispatch=False, fuse_combine=False):
    """Run the layer through the C ABI; return (cfg, inputs, outputs, ws).
    An ``inp["sel_bias"]`` routes with the selection-only bias; ``health``
    also asks for the routing-health indicators; ``fuse_dispatch`` runs the
    first GEMM on gathered token rows (no xd); ``fuse_combine`` runs the
    combine inside the second GEMM."""
    if inp is None:
        inp = inputs.make_inputs(wl, "cuda", expert_bias=expert_bias)
    cfg = moe.config_from_workload(wl, write_logits=True, reroute=reroute,
                                   fuse_dispatch=fuse_dispatch, fuse_combine=fuse_combine)
    ws = moe.workspace(cfg)
    out = moe.allocate(cfg, health=health)
    if stages:
        moe.forward_stages(cfg, inp, out, ws, alpha)
    else:
        moe.forward(cfg, inp, out, ws, alpha)
    torch.cuda.synchronize()
    assert moe.device_status(ws) == moe.MOE_OK
    return cfg, inp, out, ws


def tail_class(n_rows):
    """Which tile shape covers an expert's last rows in the pair-body/tail
    split of the tensor-core GEMM: 'whole' (rows % 256 == 0, only 256-row
    pair tiles), 'tail' (1..128 rows left: a one-CTA 128-row tile) or
    'pair_part' (129..255 left: a partly filled pair tile)."""
    m = int(n_rows) % 256
    return "whole" if m == 0 else ("tail" if m <= 128 else "pair_part")


def sample_rows(offsets, E, per_expert=6, max_experts=None, seed=0, per_class=None):
    """Rows of the dispatch buffer to check: each chosen expert's first and
    last rows, the rows around the 128- and 256-row tile edges (including the
    edges of its last, partial tile), and a few random ones.  ``per_class``
    picks up to that many experts of each tail_class before the random ones
    (so every tile shape of the GEMM's split is covered)."""
    rng = np.random.default_rng(seed)
    experts = [e for e in range(E) if offsets[e + 1] > offsets[e]]
    if max_experts is not None and len(experts) > max_experts:
        keep = {experts[0], experts[-1]}
        if per_class:
            for cls in ("whole", "tail", "pair_part"):
                of = [e for e in experts if tail_class(offsets[e + 1] - offsets[e]) == cls]
                if of:
                    keep |= set(rng.choice(of, min(per_class, len(of)), replace=False).tolist())
        rest = [e for e in experts if e not in keep]
        n_more = max(0, min(len(rest), max_experts - len(keep)))
        if n_more:
            keep |= set(rng.choice(rest, n_more, replace=False).tolist())
        experts = sorted(keep)
    rows = set()
    for e in experts:
        a, b = int(offsets[e]), int(offsets[e + 1])
        last_tile = a + ((b - a - 1) // 256) * 256
        for r in (a, b - 1, a + 127, a + 128, a + 255, a + 256, last_tile - 1, last_tile,
                  last_tile + 127, last_tile + 128):
            if a <= r < b:
                rows.add(r)
        for r in rng.integers(a, b, size=min(per_expert, b - a)):
            rows.add(int(r))
    return np.array(sorted(rows), np.int32)


def oracle_yd(wl, inp, xd_rows, rows, offsets, experts_per_copy=16):
    """Oracle expert outputs for the given buffer rows (device xd row values),
    copying to the host only the experts those rows belong to, a group of at
    most ``experts_per_copy`` experts at a time (bounded host memory)."""
    E = wl.E
    rows = np.asarray(rows)
    exp_of = np.searchsorted(offsets, rows, side="right") - 1
    experts = np.unique(exp_of)
    assert E >= len(experts)
    out = np.empty((len(rows), wl.d), np.float64)
    for g0 in range(0, len(experts), experts_per_copy):
        grp = experts[g0:g0 + experts_per_copy]
        sel = np.nonzero(np.isin(exp_of, grp))[0]
        sub_off = np.searchsorted(exp_of[sel], grp, side="left").tolist() + [len(sel)]
        sub_off = np.array(sub_off, np.int32)
        idx = torch.as_tensor(grp, device=inp["W1"].device, dtype=torch.long)
        W1 = h(inp["W1"].index_select(0, idx))
        W2 = h(inp["W2"].index_select(0, idx))
        b1 = h(inp["b1"].index_select(0, idx))
        b2 = h(inp["b2"].index_select(0, idx))
        out[sel] = oracle.ffn_rows(xd_rows[sel], sub_off, W1, b1, W2, b2, ACT[wl.act])
    return out


def check_forward(wl, inp, out, alpha=1.0, full=False, max_rows_check=None, n_tokens=None,
                  max_experts=None, e2e_tokens=64, seed=0, reroute=False, per_expert=6,
                  per_class=None):
    """Compare every output of one forward pass with the oracle (routing with
    inp["sel_bias"] when present; out["health"] when present)."""
    sel_bias = h(inp["sel_bias"]) if inp.get("sel_bias") is not None else None
    T, E, k, d = wl.T, wl.E, wl.k, wl.d
    x = h(inp["x"])
    Wr, br = h(inp["Wr"]), h(inp["br"])
    rng = np.random.default_rng(seed)

    # 1. logits (oracle router in double), on all or sampled tokens
    logits = h(out["logits"])
    if full or n_tokens is None:
        tok_l = np.arange(T)
    else:
        tok_l = np.unique(np.concatenate([[0, T - 1], rng.choice(T, min(n_tokens, T), False)]))
    ref_logits = oracle.router_logits(x[tok_l], Wr, br)
    assert_rel_rms(logits[tok_l], ref_logits, 1e-5, "logits")

    # 2. selection on the device's own logits: ids bit-exact, weights, psum
    ids_ref, w_ref, psum_ref, _, cand_ref = oracle.select(logits, k, wl.renormalize,
                                                          sel_bias=sel_bias, want_cand=True)
    np.testing.assert_array_equal(h(out["topk_ids"]), ids_ref, "topk_ids")
    assert_rel_rms(h(out["topk_w"]), w_ref, 1e-4, "topk_w")
    assert_rel_rms(h(out["psum"]), psum_ref, 1e-4, "psum")

    # 3. capacity fill: every index bit-exact
    C = oracle.capacity(T, k, E, wl.capacity_factor)
    fl = oracle.fill_reroute(ids_ref, cand_ref, E, C) if reroute else oracle.fill(ids_ref, E, C)
    for name in ["counts", "kept", "offsets", "slot_row"]:
        np.testing.assert_array_equal(h(out[name]), fl[name], name)
    n = int(fl["offsets"][E])
    np.testing.assert_array_equal(h(out["row_token"])[:n], fl["row_token"], "row_token")

    # 4. permutation: xd rows are the token rows, bit for bit.  Rows checked:
    # all, or a stratified sample plus every kept row of a few sampled tokens
    # (those tokens then get an end-to-end check in step 7).
    if full:
        rows = np.arange(n, dtype=np.int32)
        toks = np.arange(T, dtype=np.int64)
    else:
        rows = sample_rows(fl["offsets"], E, per_expert=per_expert, max_experts=max_experts,
                           seed=seed, per_class=per_class)
        if max_rows_check is not None and len(rows) > max_rows_check:
            rows = np.sort(rng.choice(rows, max_rows_check, replace=False)).astype(np.int32)
        toks = np.sort(rng.choice(T, min(e2e_tokens, T), replace=False)).astype(np.int64)
        tr = fl["slot_row"][toks].reshape(-1)
        rows = np.union1d(rows, tr[tr >= 0]).astype(np.int32)
    ridx = torch.as_tensor(rows, device="cuda", dtype=torch.long)
    if out.get("xd") is not None:
        xd_rows = h(out["xd"].index_select(0, ridx)) if len(rows) else x[:0]
        np.testing.assert_array_equal(xd_rows, x[fl["row_token"][rows]], "xd")
    else:  # fused dispatch: the first GEMM read the token rows themselves
        xd_rows = x[fl["row_token"][rows]]

    # 5. expert FFN on those rows
    yd_ref = oracle_yd(wl, inp, xd_rows, rows, fl["offsets"]) if len(rows) else None
    yd_rows = f64(out["yd"].index_select(0, ridx)) if len(rows) else None
    if len(rows):
        assert_float(yd_rows, yd_ref, wl.dtype, "yd")

    # 6. combine from the device's yd (isolates the combine kernel): all
    # tokens, or a sample of tokens (only their rows of yd are copied back)
    def y_rows(tk):
        return f64(out["y"].index_select(0, torch.as_tensor(tk, device="cuda", dtype=torch.long)))

    w_dev = h(out["topk_w"]).astype(np.float64)
    if full or T <= 4096:
        ct = np.arange(T, dtype=np.int64)
    else:
        ct = np.sort(rng.choice(T, 4096, replace=False)).astype(np.int64)
    cr = fl["slot_row"][ct].reshape(-1)
    cr = np.unique(cr[cr >= 0]).astype(np.int64)
    cidx = torch.as_tensor(cr, device="cuda", dtype=torch.long)
    yd_c = f64(out["yd"].index_select(0, cidx)) if len(cr) else np.zeros((0, d))
    c_index = np.full(n + 1, -1, np.int64)
    c_index[cr] = np.arange(len(cr))
    y_from_dev = oracle.combine(fl["slot_row"], w_dev, yd_c, d, tokens=ct, row_index=c_index)
    assert_float(y_rows(ct), y_from_dev, wl.dtype, "y (combine of device yd)")

    # 7. end to end on the sampled tokens (all of their kept rows were checked)
    if len(toks):
        row_index = np.full(n + 1, -1, np.int64)
        row_index[rows] = np.arange(len(rows))
        y_ref = oracle.combine(fl["slot_row"], w_ref, yd_ref if yd_ref is not None else
                               np.zeros((0, d)), d, tokens=toks, row_index=row_index)
        assert_float(y_rows(toks), y_ref, wl.dtype, "y (end to end)")

    # 8. statistics
    f_ref, pbar_ref, l_ref = oracle.aux(fl["counts"], psum_ref, T, alpha)
    assert_rel_rms(h(out["f"]), f_ref, 1e-6, "f")
    assert_rel_rms(h(out["pbar"]), pbar_ref, 1e-4, "pbar")
    assert abs(float(h(out["l_aux"])[0]) - l_ref) <= 1e-4 * abs(l_ref) + 1e-7

    # 9. routing health
    if out.get("health") is not None:
        ref = oracle.routing_health(fl["counts"], fl["kept"], T, k)
        np.testing.assert_allclose(h(out["health"]), ref, rtol=1e-4, atol=1e-6,
                                   err_msg="health")
    exp_of = np.searchsorted(fl["offsets"], rows, side="right") - 1
    return dict(n_rows=n, rows_checked=len(rows), tokens_e2e=len(toks),
                experts_checked=len(np.unique(exp_of)) if len(rows) else 0,
                classes_checked=sorted({tail_class(fl["kept"][e]) for e in np.unique(exp_of)})
                if len(rows) else [])
