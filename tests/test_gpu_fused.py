"""The permutation folded into the first expert GEMM (moe_ffn_up_gather,
cfg.fuse_dispatch) and the combine folded into the second one
(moe_ffn_down_combine, cfg.fuse_combine): the fused permutation/dispatch and
combine kernels of [MoE Gate 分布式通信 mianshidashi, 06].  Each case runs the
layer on the same inputs through the materialised path (dispatch buffer xd,
separate combine) and through the fused one(s), and requires every output to
be identical bit for bit (a GEMM row depends only on its own A row; the
fused combine sums the same bf16 rows in the same order); the fused run is
also checked against the oracle."""

import os

import numpy as np
import pytest
import torch

from routing_dispatch_expert_06_b300 import build, inputs, moe

from parity import check_forward, h, run_gpu

pytestmark = pytest.mark.gpu

W = inputs.WORKLOADS

OUTPUTS = ["logits", "topk_ids", "topk_w", "psum", "counts", "kept", "offsets", "slot_row",
           "f", "pbar", "l_aux", "y"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    moe.load()


def same_as_materialised(wl, expert_bias=False, reroute=False, stages=False,
                         fuse_dispatch=True, fuse_combine=False, inp=None):
    if inp is None:
        inp = inputs.make_inputs(wl, "cuda", expert_bias=expert_bias)
    _, _, out_m, _ = run_gpu(wl, inp=inp, reroute=reroute)
    _, _, out_f, _ = run_gpu(wl, inp=inp, reroute=reroute, stages=stages,
                             fuse_dispatch=fuse_dispatch, fuse_combine=fuse_combine)
    assert (out_f["xd"] is None) == fuse_dispatch
    for name in OUTPUTS:
        assert torch.equal(out_m[name], out_f[name]), name
    n = int(h(out_m["offsets"])[-1])
    for name in ["row_token", "H", "yd"]:
        assert torch.equal(out_m[name][:n], out_f[name][:n]), name
    return inp, out_f


CASES = {
    # 8 experts, 8192 rows: CTA pairs, whole 256-row tiles
    "t4096_d1024_e8_top2": dict(wl=W["bf16_t4096_d1024_e8_top2"], e2e_tokens=256),
    # Zipf-skewed 64 experts, ragged groups and empty experts
    "t3000_d2048_e64_top6": dict(wl=W["bf16_t8192_d2048_e64_top6"].replace(T=3000),
                                 e2e_tokens=64),
    # K = d = 1000: the last 64-column block holds 40 columns (zero-filled
    # pieces past K); capacity below demand so that slots are dropped
    "t2000_d1000_e8_top2_ragged_k": dict(
        wl=W["bf16_t4096_d1024_e8_top2"].replace(T=2000, d=1000, d_ff=512,
                                                 capacity_factor=0.8),
        e2e_tokens=128),
    # K = d = 960: 15 64-wide k-blocks, so the last pipeline stage of two
    # holds one (the gathering producer copies no k-block past K); the
    # second GEMM's K = d_ff = 704 has 11
    "t1500_d960_e8_top2_odd_k": dict(
        wl=W["bf16_t4096_d1024_e8_top2"].replace(T=1500, d=960, d_ff=704), e2e_tokens=128),
    # 256 experts: pair launch on whole 256-row tiles plus the overlapped
    # one-CTA tail launch, every remainder size
    "t12000_d256_e256_top8_tail": dict(
        wl=W["bf16_t32768_d7168_e256_top8"].replace(T=12000, d=256, d_ff=512,
                                                    capacity_factor=2.0),
        e2e_tokens=64, expert_bias=True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_fused_dispatch_equals_materialised_and_oracle(name):
    case = dict(CASES[name])
    wl = case.pop("wl")
    e2e = case.pop("e2e_tokens")
    inp, out = same_as_materialised(wl, expert_bias=case.get("expert_bias", False))
    check_forward(wl, inp, out, n_tokens=512, e2e_tokens=e2e, max_experts=12,
                  max_rows_check=400)


def test_fused_dispatch_one_sm_gemm():
    wl = CASES["t3000_d2048_e64_top6"]["wl"]
    os.environ["MOE_GEMM_PAIR"] = "0"
    try:
        same_as_materialised(wl)
    finally:
        del os.environ["MOE_GEMM_PAIR"]


def test_fused_dispatch_stage_calls_and_reroute():
    wl = W["bf16_t4096_d1024_e8_top2"].replace(T=2048, capacity_factor=0.75)
    same_as_materialised(wl, stages=True)
    inp, out = same_as_materialised(wl, reroute=True)
    check_forward(wl, inp, out, n_tokens=256, e2e_tokens=64, reroute=True)


def test_fused_dispatch_unsupported_on_decode_sizes():
    wl = W["decode_bf16_t8_d2048_e64_top6"]
    cfg = moe.config_from_workload(wl, fuse_dispatch=True)
    inp = inputs.make_inputs(wl, "cuda")
    out = moe.allocate(cfg)
    ws = moe.workspace(cfg)
    with pytest.raises(moe.MoeError) as e:
        moe.forward(cfg, inp, out, ws, 1.0)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert moe.device_status(ws) == moe.MOE_OK


# ---- combine folded into the second GEMM ----

@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("with_gather", [False, True], ids=["xd", "gather"])
def test_fused_combine_equals_materialised_and_oracle(name, with_gather):
    case = dict(CASES[name])
    wl = case.pop("wl")
    e2e = case.pop("e2e_tokens")
    inp, out = same_as_materialised(wl, expert_bias=case.get("expert_bias", False),
                                    fuse_dispatch=with_gather, fuse_combine=True)
    check_forward(wl, inp, out, n_tokens=512, e2e_tokens=e2e, max_experts=12,
                  max_rows_check=400)


def test_fused_combine_one_sm_gemm_and_stage_calls():
    wl = CASES["t3000_d2048_e64_top6"]["wl"]
    os.environ["MOE_GEMM_PAIR"] = "0"
    try:
        same_as_materialised(wl, fuse_dispatch=False, fuse_combine=True)
    finally:
        del os.environ["MOE_GEMM_PAIR"]
    same_as_materialised(wl, fuse_dispatch=False, fuse_combine=True, stages=True)


def test_fused_combine_zeroes_fully_dropped_tokens_and_reroutes():
    # A capacity far below demand: the first-come fill leaves many late tokens
    # with no kept slot, whose y must be exactly 0 (no arrival ever comes for
    # them); also with the overflow reroute.
    wl = inputs.Workload("drops_fused", 4000, 256, 512, 16, 4, 0.3, True, "gelu_tanh", "bf16",
                         23, "zipf:0.8")
    inp, out = same_as_materialised(wl, fuse_dispatch=False, fuse_combine=True)
    dropped = (h(out["slot_row"]) < 0).all(axis=1)
    assert dropped.sum() > 100
    assert (inputs.as_f64(h(out["y"]))[dropped] == 0).all()
    check_forward(wl, inp, out, full=True)
    inp, out = same_as_materialised(wl, fuse_dispatch=False, fuse_combine=True, reroute=True,
                                    inp=inp)
    check_forward(wl, inp, out, full=True, reroute=True)


def test_fused_combine_counters_return_to_zero_between_calls():
    # Two different routings through one workspace, back to back (and a
    # third call repeating the first): each y equals the materialised path's,
    # so no arrival count survives a call.
    wl = W["bf16_t8192_d2048_e64_top6"].replace(T=3000)
    cfg = moe.config_from_workload(wl, write_logits=True, fuse_combine=True)
    ws = moe.workspace(cfg)
    out = moe.allocate(cfg)
    inps = [inputs.make_inputs(wl, "cuda", seed=s) for s in (wl.seed, wl.seed + 5)]
    refs = []
    for inp in inps:
        _, _, ref, _ = run_gpu(wl, inp=inp)
        refs.append(ref)
    for i in (0, 1, 0):
        out["y"].fill_(7.0)
        moe.forward(cfg, inps[i], out, ws, 1.0)
        torch.cuda.synchronize()
        assert moe.device_status(ws) == moe.MOE_OK
        assert torch.equal(out["y"], refs[i]["y"]), i


def test_fused_combine_needs_its_flag_and_is_unsupported_on_decode_sizes():
    wl = W["decode_bf16_t8_d2048_e64_top6"]
    cfg = moe.config_from_workload(wl, fuse_combine=True)
    inp = inputs.make_inputs(wl, "cuda")
    out = moe.allocate(cfg)
    ws = moe.workspace(cfg)
    with pytest.raises(moe.MoeError) as e:
        moe.forward(cfg, inp, out, ws, 1.0)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED
    wl = W["bf16_t4096_d1024_e8_top2"].replace(T=512)
    cfg = moe.config_from_workload(wl)  # fuse_combine = 0: no counters in the workspace
    ws = moe.workspace(cfg)
    out = moe.allocate(cfg)
    with pytest.raises(moe.MoeError) as e:
        moe.ffn_down_combine(cfg, out["H"], out["offsets"], out["row_token"], out["slot_row"],
                             out["topk_w"], inp["W2"], inp["b2"], out["yd"], out["y"], ws)
    assert e.value.code == moe.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
