"""Router parity on ragged shapes, through the C ABI (moe_route).

Three routers are checked: the warp router (bf16, E <= 32, the default there),
the tensor-core router (bf16, E <= 256) and the generic CUDA-core router
(MOE_ROUTE_IMPL=warp|tc|simt forces one where it applies).  Against the
oracle ("MoE 模型原理" §2.1–§2.2):

* logits within 1e-5 · max(|ref|, rms(row)) of the double-precision router;
* top-k ids bit-exact with the oracle's selection on the device's own fp32
  logits (so both sides rank the same numbers), weights and Σ_t p within 1e-4.

Shapes cover a ragged last token tile, d not a multiple of the 64-wide
k-block, E not a multiple of 16, E = 1, k = E, k = 16, the widest E (256),
and exact ties (equal logits must go to the lower expert index).
"""

import os

import numpy as np
import pytest
import torch

import oracle
from routing_dispatch_expert_06_b300 import build, inputs, moe

from parity import assert_rel_rms, h

pytestmark = pytest.mark.gpu

# (T, d, E, k, renormalize, router bias)
CASES = [
    (300, 200, 20, 3, True, "normal:1.0"),
    (129, 72, 1, 1, True, "zero"),
    (1000, 520, 256, 16, False, "normal:1.0"),
    (64, 64, 16, 16, True, "zipf:0.8"),
    (5000, 1024, 8, 2, True, "zero"),
    (777, 7168, 256, 8, False, "normal:1.0"),
    (2, 8, 3, 2, True, "linear_skew"),
    (4097, 2048, 64, 6, True, "zipf:0.8"),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    moe.load()


def _workload(T, d, E, k, renorm, bias, seed=11):
    return inputs.Workload(f"route_t{T}_d{d}_e{E}_top{k}", T, d, 8, E, k, 1.0, renorm,
                           "gelu_tanh", "bf16", seed, bias)


def _route(wl, inp, impl):
    cfg = moe.config_from_workload(wl, write_logits=True)
    ws = moe.workspace(cfg)
    out = moe.allocate(cfg)
    os.environ["MOE_ROUTE_IMPL"] = impl
    try:
        moe.route(cfg, inp["x"], inp["Wr"], inp["br"], out, ws)
        torch.cuda.synchronize()
    finally:
        os.environ.pop("MOE_ROUTE_IMPL", None)
    assert moe.device_status(ws) == moe.MOE_OK
    return out


def _check(wl, inp, out):
    logits = h(out["logits"])
    ref = oracle.router_logits(h(inp["x"]), h(inp["Wr"]), h(inp["br"]))
    assert_rel_rms(logits, ref, 1e-5, "logits")
    ids, w, psum, _ = oracle.select(logits, wl.k, wl.renormalize)
    np.testing.assert_array_equal(h(out["topk_ids"]), ids, "topk_ids")
    assert_rel_rms(h(out["topk_w"]), w, 1e-4, "topk_w")
    assert_rel_rms(h(out["psum"]), psum, 1e-4, "psum")


@pytest.mark.parametrize("impl", ["warp", "tc", "simt"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"t{c[0]}_d{c[1]}_e{c[2]}_k{c[3]}")
def test_router_matches_oracle(case, impl):
    wl = _workload(*case)
    inp = inputs.make_inputs(wl, "cuda")
    _check(wl, inp, _route(wl, inp, impl))


@pytest.mark.parametrize("impl", ["warp", "tc", "simt"])
def test_router_ties_go_to_lower_index(impl):
    # W_r = 0 makes every logit equal to its bias; the bias repeats values, so
    # the ranking must break ties by the lower expert index.
    T, d, E, k = 200, 128, 24, 5
    wl = _workload(T, d, E, k, True, "zero")
    inp = inputs.make_inputs(wl, "cuda")
    inp["Wr"].zero_()
    inp["br"].copy_(torch.tensor([0.5, 1.0, 1.0, 0.25, 1.0, 0.5] * 4, device="cuda"))
    out = _route(wl, inp, impl)
    ids = h(out["topk_ids"])
    assert (ids == np.array([1, 2, 4, 7, 8], np.int32)).all()
    _check(wl, inp, out)
    np.testing.assert_allclose(h(out["topk_w"]), 0.2, rtol=1e-6)


def test_tensor_core_router_agrees_with_cuda_core_router():
    wl = _workload(3000, 2048, 64, 6, True, "zipf:0.8", seed=5)
    inp = inputs.make_inputs(wl, "cuda")
    a = _route(wl, inp, "tc")
    b = _route(wl, inp, "simt")
    la, lb = h(a["logits"]), h(b["logits"])
    assert_rel_rms(la, lb.astype(np.float64), 2e-5, "tc vs simt logits")
    same = (h(a["topk_ids"]) == h(b["topk_ids"])).all(axis=1)
    # the two routers round differently, so a near-tie may rank differently;
    # with these seeded inputs nearly every token must agree
    assert same.mean() > 0.99


def test_warp_router_agrees_with_tensor_core_router():
    wl = _workload(5000, 1024, 8, 2, True, "normal:0.5", seed=9)
    inp = inputs.make_inputs(wl, "cuda")
    a = _route(wl, inp, "warp")
    b = _route(wl, inp, "tc")
    assert_rel_rms(h(a["logits"]), h(b["logits"]).astype(np.float64), 2e-5, "warp vs tc logits")
    same = (h(a["topk_ids"]) == h(b["topk_ids"])).all(axis=1)
    assert same.mean() > 0.99


def test_unaligned_inputs_take_the_generic_router():
    # x starting 2 bytes past a 16-byte boundary: the 16-byte routers must not
    # be used; the result still matches the oracle.
    wl = _workload(300, 200, 20, 3, True, "normal:1.0")
    inp = inputs.make_inputs(wl, "cuda")
    buf = torch.empty(wl.T * wl.d + 1, dtype=torch.bfloat16, device="cuda")
    x = buf[1:].view(wl.T, wl.d)
    x.copy_(inp["x"])
    assert x.data_ptr() % 16 != 0
    inp = dict(inp, x=x)
    _check(wl, inp, _route(wl, inp, "warp"))


@pytest.mark.parametrize("case", [(8, 7168, 256, 8), (3000, 1024, 64, 6), (5000, 256, 8, 2)],
                         ids=lambda c: f"t{c[0]}_e{c[2]}")
def test_column_sums_repeat_exactly_and_match_the_whole_layer(case):
    # The tensor-core router keeps Σ_t p as integer sums in the workspace and
    # clears them after use: repeated calls give the same bits, and the whole
    # layer (which converts them in the dispatch) gives the same psum.
    T, d, E, k = case
    wl = inputs.Workload(f"psum_t{T}_e{E}", T, d, 64, E, k, 1.0, True, "gelu_tanh", "bf16", 3,
                         "normal:1.0")
    inp = inputs.make_inputs(wl, "cuda")
    cfg = moe.config_from_workload(wl)
    ws = moe.workspace(cfg)
    out = moe.allocate(cfg)
    runs = []
    for _ in range(3):
        moe.route(cfg, inp["x"], inp["Wr"], inp["br"], out, ws)
        torch.cuda.synchronize()
        runs.append(h(out["psum"]).copy())
    assert moe.device_status(ws) == moe.MOE_OK
    for r in runs[1:]:
        np.testing.assert_array_equal(r.view(np.uint32), runs[0].view(np.uint32))
    moe.forward(cfg, inp, out, ws, 0.01)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(h(out["psum"]).view(np.uint32), runs[0].view(np.uint32))
    ref_logits = oracle.router_logits(h(inp["x"]), h(inp["Wr"]), h(inp["br"]))
    _, _, psum, _ = oracle.select(ref_logits, k, True)
    assert_rel_rms(runs[0], psum, 1e-4, "psum")


def _route_sel(wl, inp, impl, sel_bias):
    cfg = moe.config_from_workload(wl, write_logits=True)
    ws = moe.workspace(cfg)
    out = moe.allocate(cfg)
    os.environ["MOE_ROUTE_IMPL"] = impl
    try:
        moe.route(cfg, inp["x"], inp["Wr"], inp["br"], out, ws, sel_bias=sel_bias)
        torch.cuda.synchronize()
    finally:
        os.environ.pop("MOE_ROUTE_IMPL", None)
    assert moe.device_status(ws) == moe.MOE_OK
    return out


@pytest.mark.parametrize("impl", ["warp", "tc", "simt"])
@pytest.mark.parametrize("case", [(300, 200, 20, 3, True), (5000, 1024, 8, 2, True),
                                  (1000, 520, 256, 16, False), (4097, 2048, 64, 6, True),
                                  (9, 7168, 256, 8, False)],
                         ids=lambda c: f"t{c[0]}_e{c[2]}_k{c[3]}")
def test_selection_bias_matches_oracle(case, impl):
    # Experts are ranked by logit + sel_bias (fp32); the weights, Σp and
    # logits stay the unbiased ones.  The bias must change many choices.
    T, d, E, k, renorm = case
    wl = _workload(T, d, E, k, renorm, "normal:1.0", seed=13)
    inp = inputs.make_inputs(wl, "cuda")
    sb = torch.randn(E, generator=torch.Generator("cuda").manual_seed(7), device="cuda") * 1.5
    out = _route_sel(wl, inp, impl, sb)
    logits = h(out["logits"])
    ids, w, psum, _ = oracle.select(logits, k, renorm, sel_bias=h(sb))
    np.testing.assert_array_equal(h(out["topk_ids"]), ids, "topk_ids")
    assert_rel_rms(h(out["topk_w"]), w, 1e-4, "topk_w")
    assert_rel_rms(h(out["psum"]), psum, 1e-4, "psum")
    plain, *_ = oracle.select(logits, k, renorm)
    if T > 100:
        assert (plain != ids).any(axis=1).mean() > 0.1


@pytest.mark.parametrize("impl", ["warp", "tc", "simt"])
def test_selection_bias_ties_go_to_lower_index(impl):
    # W_r = 0 and b_r = 0: every logit is 0, so the keys are the bias, which
    # repeats values; equal keys must go to the lower expert index, and the
    # weights are the unbiased uniform 1/k.
    T, d, E, k = 200, 128, 24, 5
    wl = _workload(T, d, E, k, True, "zero")
    inp = inputs.make_inputs(wl, "cuda")
    inp["Wr"].zero_()
    sb = torch.tensor([0.5, 1.0, 1.0, 0.25, 1.0, 0.5] * 4, device="cuda")
    out = _route_sel(wl, inp, impl, sb)
    assert (h(out["topk_ids"]) == np.array([1, 2, 4, 7, 8], np.int32)).all()
    np.testing.assert_allclose(h(out["topk_w"]), 0.2, rtol=1e-6)


# With 75 or more 128-token tiles each CTA of the tensor-core router reduces a
# whole tile (one split over d), so the selection kernel reads one partial per
# token.  Every lane layout of the selection at that size: E <= 8 (8 lanes per
# token), <= 16, <= 32, 64 (2 columns per lane), 100 (4), 130 and 256 (8); a
# ragged last tile, d not a multiple of 64, k = 12 = E and k = 16.
ONE_SPLIT_CASES = [
    (9601, 520, 256, 16, False, "normal:1.0"),
    (12000, 1024, 8, 2, True, "zero"),
    (9500, 136, 12, 12, True, "zipf:0.8"),
    (10000, 200, 20, 3, True, "normal:1.0"),
    (9999, 2048, 64, 6, True, "zipf:0.8"),
    (9700, 256, 100, 4, False, "normal:1.0"),
    (9700, 256, 130, 5, True, "normal:1.0"),
    # E > 128: CTA pairs on 256-token tiles; T = 38·256 + 50, so the last
    # tile's odd CTA has no token (its copies read zeros past T)
    (9778, 200, 200, 8, False, "normal:1.0"),
]


@pytest.mark.parametrize("case", ONE_SPLIT_CASES,
                         ids=lambda c: f"t{c[0]}_d{c[1]}_e{c[2]}_k{c[3]}")
def test_one_split_router_matches_oracle(case):
    wl = _workload(*case)
    inp = inputs.make_inputs(wl, "cuda")
    _check(wl, inp, _route(wl, inp, "tc"))


@pytest.mark.parametrize("case", [(9601, 520, 256, 8, False), (12000, 512, 8, 2, True),
                                  (9999, 1024, 64, 6, True)],
                         ids=lambda c: f"t{c[0]}_e{c[2]}_k{c[3]}")
def test_one_split_router_with_selection_bias(case):
    T, d, E, k, renorm = case
    wl = _workload(T, d, E, k, renorm, "normal:1.0", seed=13)
    inp = inputs.make_inputs(wl, "cuda")
    sb = torch.randn(E, generator=torch.Generator("cuda").manual_seed(7), device="cuda") * 1.5
    out = _route_sel(wl, inp, "tc", sb)
    logits = h(out["logits"])
    ids, w, psum, _ = oracle.select(logits, k, renorm, sel_bias=h(sb))
    np.testing.assert_array_equal(h(out["topk_ids"]), ids, "topk_ids")
    assert_rel_rms(h(out["topk_w"]), w, 1e-4, "topk_w")
    assert_rel_rms(h(out["psum"]), psum, 1e-4, "psum")
    plain, *_ = oracle.select(logits, k, renorm)
    assert (plain != ids).any(axis=1).mean() > 0.1


def test_one_split_router_breaks_ties_by_lower_index():
    T, d, E, k = 9700, 128, 24, 5
    wl = _workload(T, d, E, k, True, "zero")
    inp = inputs.make_inputs(wl, "cuda")
    inp["Wr"].zero_()
    inp["br"].copy_(torch.tensor([0.5, 1.0, 1.0, 0.25, 1.0, 0.5] * 4, device="cuda"))
    out = _route(wl, inp, "tc")
    assert (h(out["topk_ids"]) == np.array([1, 2, 4, 7, 8], np.int32)).all()
    np.testing.assert_allclose(h(out["topk_w"]), 0.2, rtol=1e-6)
    _check(wl, inp, out)


def test_one_split_router_repeats_column_sums_exactly():
    # Integer column sums give the same bits on every call, and the whole
    # layer (which converts them in the dispatch) agrees; ids repeat too.
    wl = inputs.Workload("psum_fused", 10000, 512, 64, 64, 6, 1.0, True, "gelu_tanh", "bf16", 3,
                         "normal:1.0")
    inp = inputs.make_inputs(wl, "cuda")
    cfg = moe.config_from_workload(wl)
    ws = moe.workspace(cfg)
    out = moe.allocate(cfg)
    runs = []
    for _ in range(3):
        moe.route(cfg, inp["x"], inp["Wr"], inp["br"], out, ws)
        torch.cuda.synchronize()
        runs.append((h(out["psum"]).copy(), h(out["topk_ids"]).copy()))
    assert moe.device_status(ws) == moe.MOE_OK
    for p, i in runs[1:]:
        np.testing.assert_array_equal(p.view(np.uint32), runs[0][0].view(np.uint32))
        np.testing.assert_array_equal(i, runs[0][1])
    moe.forward(cfg, inp, out, ws, 0.01)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(h(out["psum"]).view(np.uint32), runs[0][0].view(np.uint32))
    ref_logits = oracle.router_logits(h(inp["x"]), h(inp["Wr"]), h(inp["br"]))
    _, _, psum, _ = oracle.select(ref_logits, wl.k, True)
    assert_rel_rms(runs[0][0], psum, 1e-4, "psum")
