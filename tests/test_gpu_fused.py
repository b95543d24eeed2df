"""The permutation folded into the first expert GEMM (moe_ffn_up_gather,
cfg.fuse_dispatch): the fused permutation/dispatch kernel of [MoE Gate
分布式通信 mianshidashi, 06].  Each case runs the layer twice on the same
inputs, once through the dispatch buffer xd and once gathering the token rows
inside the GEMM, and requires every output to be identical bit for bit (a
GEMM row depends only on its own A row); the fused run is also checked
against the oracle."""

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


def same_as_materialised(wl, expert_bias=False, reroute=False, stages=False):
    inp = inputs.make_inputs(wl, "cuda", expert_bias=expert_bias)
    _, _, out_m, _ = run_gpu(wl, inp=inp, reroute=reroute)
    _, _, out_f, _ = run_gpu(wl, inp=inp, reroute=reroute, stages=stages, fuse_dispatch=True)
    assert out_f["xd"] is None
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
