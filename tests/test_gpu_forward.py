"""Parity of the CUDA path (through the C ABI) with the CPU oracle on the
seeded workloads, at full size.  Integer outputs are compared bit for bit,
floats within the tolerances stated in tests/parity.py."""

import os

import numpy as np
import pytest
import torch

from routing_dispatch_expert_06_b300 import build, inputs, moe

from parity import check_forward, h, run_gpu

pytestmark = pytest.mark.gpu

W = inputs.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    moe.load()


def test_fp32_t512_full():
    wl = W["fp32_t512_d128_e8_top2"]
    _, inp, out, _ = run_gpu(wl)
    info = check_forward(wl, inp, out, full=True)
    assert info["n_rows"] < wl.T * wl.k  # the skewed router bias makes experts overflow


def test_bf16_t4096_d1024_e8_top2():
    wl = W["bf16_t4096_d1024_e8_top2"]
    _, inp, out, _ = run_gpu(wl)
    check_forward(wl, inp, out, e2e_tokens=256)


def test_bf16_t8192_d2048_e64_top6():
    wl = W["bf16_t8192_d2048_e64_top6"]
    _, inp, out, _ = run_gpu(wl)
    info = check_forward(wl, inp, out, e2e_tokens=64)
    assert info["n_rows"] < wl.T * wl.k  # Zipf bias: hot experts overflow


def test_bf16_t16384_d4096_e8_top1():
    wl = W["bf16_t16384_d4096_e8_top1"]
    _, inp, out, _ = run_gpu(wl)
    info = check_forward(wl, inp, out, n_tokens=2048, e2e_tokens=256, max_rows_check=400)
    assert info["tokens_e2e"] >= 256
    # the dispatch buffer is in expert order, so the four groups of two
    # experts are contiguous: group g = rows offsets[2g] .. offsets[2g+2]
    off = h(out["offsets"])
    assert (np.diff(off[::2]) >= 0).all()


def test_bf16_t32768_d7168_e256_top8():
    # The largest layer: 64 tokens end to end (every kept row of theirs), and
    # over 1000 expert-output rows from at least 48 experts, at least four
    # experts of each tile shape of the GEMM's pair-body/tail split (rows % 256
    # = 0; 1..128; 129..255) with the rows at every tile edge.
    wl = W["bf16_t32768_d7168_e256_top8"]
    _, inp, out, _ = run_gpu(wl)
    info = check_forward(wl, inp, out, n_tokens=384, e2e_tokens=64, max_experts=56,
                         per_expert=12, per_class=6)
    assert info["tokens_e2e"] >= 64
    assert info["rows_checked"] >= 1000 and info["experts_checked"] >= 48
    assert info["classes_checked"] == ["pair_part", "tail", "whole"]


def test_fp32_gelu_full():
    # The CUDA-core (fp32) expert GEMM with the tanh-form GELU, every output
    # at the fp32 bar.
    wl = W["fp32_t512_d128_e8_top2"].replace(act="gelu_tanh")
    _, inp, out, _ = run_gpu(wl, expert_bias=True)
    check_forward(wl, inp, out, full=True)


def test_expert_bias_path():
    wl = W["bf16_t4096_d1024_e8_top2"].replace(T=1000, capacity_factor=0.9)
    _, inp, out, _ = run_gpu(wl, expert_bias=True)
    check_forward(wl, inp, out, full=True)


@pytest.mark.parametrize("extras", [False, True], ids=["plain", "sel_bias_health_reroute"])
def test_stage_calls_equal_forward_and_are_deterministic(extras):
    wl = W["bf16_t8192_d2048_e64_top6"].replace(T=3000)
    inp = inputs.make_inputs(wl, "cuda")
    if extras:
        inp["sel_bias"] = inputs.selection_bias(wl, "cuda")
    kw = dict(health=extras, reroute=extras)
    _, inp, out1, _ = run_gpu(wl, inp=inp, **kw)
    _, _, out2, _ = run_gpu(wl, inp=inp, stages=True, **kw)
    _, _, out3, _ = run_gpu(wl, inp=inp, **kw)
    n = int(h(out1["offsets"])[-1])
    names = ["logits", "topk_ids", "topk_w", "psum", "counts", "kept", "offsets",
             "slot_row", "f", "pbar", "l_aux", "y"] + (["health"] if extras else [])
    for name in names:
        for o in (out2, out3):
            assert torch.equal(out1[name], o[name]), name
    for name in ["row_token", "xd", "H", "yd"]:
        for o in (out2, out3):
            assert torch.equal(out1[name][:n], o[name][:n]), name


def test_tensor_core_gemm_matches_cuda_core_gemm():
    wl = W["bf16_t4096_d1024_e8_top2"]
    _, inp, out_tc, _ = run_gpu(wl)
    os.environ["MOE_FFN_IMPL"] = "simt"
    try:
        _, _, out_s, _ = run_gpu(wl, inp=inp)
    finally:
        del os.environ["MOE_FFN_IMPL"]
    n = int(h(out_tc["offsets"])[-1])
    a = out_tc["yd"][:n].float()
    b = out_s["yd"][:n].float()
    assert ((a - b).abs() <= 1e-2 + 2e-2 * b.abs()).all()
    ha, hb = out_tc["H"][:n].float(), out_s["H"][:n].float()
    assert ((ha - hb).abs() <= 1e-2 + 2e-2 * hb.abs()).all()


def test_two_sm_gemm_matches_one_sm_gemm():
    # Default: CTA pairs with the 2-SM MMA (M = 256); MOE_GEMM_PAIR=0 runs the
    # 1-SM kernel (M = 128).  Ragged experts with odd 128-row tile counts
    # exercise the pair's empty upper half.
    wl = W["bf16_t8192_d2048_e64_top6"].replace(T=3000)
    _, inp, out_p, _ = run_gpu(wl, expert_bias=True)
    os.environ["MOE_GEMM_PAIR"] = "0"
    try:
        _, _, out_1, _ = run_gpu(wl, inp=inp)
    finally:
        del os.environ["MOE_GEMM_PAIR"]
    n = int(h(out_p["offsets"])[-1])
    for name in ["H", "yd"]:
        a = out_p[name][:n].float()
        b = out_1[name][:n].float()
        assert ((a - b).abs() <= 1e-2 + 2e-2 * b.abs()).all(), name


@pytest.mark.parametrize("name,c", [("decode_bf16_t64_d2048_e64_top6", 1.0),
                                    ("decode_bf16_t64_d2048_e64_top6", 5.0),
                                    ("decode_bf16_t8_d7168_e256_top8", 1.25)])
def test_swapped_gemm_matches_regular_gemm(name, c):
    # With at most min(C, T·k) <= 64 rows per expert the expert GEMMs swap the
    # operands' roles (MMA M over weight rows, N over the expert's 16/32/64
    # rows); MOE_FFN_SWAP=0 runs the regular kernel.  c = 5 gives C = 30
    # (N = 32) with experts holding up to 30 rows.
    wl = W[name].replace(capacity_factor=c)
    _, inp, out_s, _ = run_gpu(wl, expert_bias=True)
    os.environ["MOE_FFN_SWAP"] = "0"
    try:
        _, _, out_r, _ = run_gpu(wl, inp=inp)
    finally:
        del os.environ["MOE_FFN_SWAP"]
    n = int(h(out_s["offsets"])[-1])
    assert n == int(h(out_r["offsets"])[-1]) > 0
    for name_ in ["H", "yd"]:
        a = out_s[name_][:n].float()
        b = out_r[name_][:n].float()
        assert ((a - b).abs() <= 1e-2 + 2e-2 * b.abs()).all(), name_


def test_forward_replays_from_a_cuda_graph():
    # moe_forward only enqueues kernels (no allocation, no synchronisation),
    # so it can be captured once and replayed; the replay must reproduce the
    # eager outputs bit for bit (the benchmark times such replays).
    wl = W["bf16_t8192_d2048_e64_top6"].replace(T=3000)
    cfg, inp, out_e, _ = run_gpu(wl)
    ws = moe.workspace(cfg)
    out_g = moe.allocate(cfg)
    moe.forward(cfg, inp, out_g, ws, 1.0)  # first call per shape: host-side setup
    torch.cuda.synchronize()
    for t in out_g.values():
        if t is not None:
            t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.forward(cfg, inp, out_g, ws, 1.0)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert moe.device_status(ws) == moe.MOE_OK
    n = int(h(out_e["offsets"])[-1])
    for name in ["logits", "topk_ids", "topk_w", "psum", "counts", "kept", "offsets", "slot_row",
                 "f", "pbar", "l_aux", "y"]:
        if out_e[name] is None:
            continue
        assert torch.equal(out_e[name], out_g[name]), name
    for name in ["row_token", "xd", "H", "yd"]:
        assert torch.equal(out_e[name][:n], out_g[name][:n]), name


def test_pair_body_and_tail_tiles_match_one_sm_gemm():
    # With E >= 128 each GEMM runs CTA pairs on whole 256-row tiles and a
    # second, overlapped one-CTA launch on every expert's last 1..128 rows.
    # Small ragged experts cover every case: no rows, < 128, 128 exactly,
    # 129..255, whole pairs plus a tail of each size.
    wl = W["bf16_t32768_d7168_e256_top8"].replace(T=12000, d=256, d_ff=512, capacity_factor=2.0)
    _, inp, out_p, _ = run_gpu(wl, expert_bias=True)
    rows = np.diff(h(out_p["offsets"]))
    assert (rows % 256 > 128).any() and ((rows % 256 > 0) & (rows % 256 <= 128)).any()
    os.environ["MOE_GEMM_PAIR"] = "0"
    try:
        _, _, out_1, _ = run_gpu(wl, inp=inp)
    finally:
        del os.environ["MOE_GEMM_PAIR"]
    n = int(h(out_p["offsets"])[-1])
    for name in ["H", "yd", "y"]:
        m = n if name != "y" else wl.T
        a = out_p[name][:m].float()
        b = out_1[name][:m].float()
        assert ((a - b).abs() <= 1e-2 + 2e-2 * b.abs()).all(), name


ODD_K_CASES = [
    # K/64 odd in both expert GEMMs (d = 960: 15 k-blocks, d_ff = 704: 11):
    # the last pipeline stage of two k-blocks holds one past K, which the copy
    # engine fills with zeros.  CTA pairs on every tile (E = 8), pairs on whole
    # 256-row tiles plus one-CTA tails (E = 256), and the swapped decode kernel.
    ("e8_pairs", W["bf16_t4096_d1024_e8_top2"].replace(T=1500, d=960, d_ff=704)),
    ("e256_pairs_and_tails", W["bf16_t32768_d7168_e256_top8"].replace(
        T=3000, d=320, d_ff=448, capacity_factor=2.0)),
    ("decode_swapped", W["decode_bf16_t8_d2048_e64_top6"].replace(d=960, d_ff=704)),
]


@pytest.mark.parametrize("name,wl", ODD_K_CASES, ids=[c[0] for c in ODD_K_CASES])
def test_odd_k_block_counts_match_oracle(name, wl):
    _, inp, out, _ = run_gpu(wl, expert_bias=True)
    check_forward(wl, inp, out, full=True)


@pytest.mark.parametrize("name", [n for n in W if n.startswith("decode_")])
def test_decode_regime(name):
    # A few tokens per call on the many-expert layers: every output is checked.
    wl = W[name]
    _, inp, out, _ = run_gpu(wl)
    check_forward(wl, inp, out, full=True)


def test_dropless_capacity_keeps_every_slot():
    # c = E/k gives C = T: no expert can overflow, so every slot is kept and
    # the buffer holds all T·k rows.
    wl = W["dropless_bf16_t8192_d2048_e64_top6"]
    _, inp, out, _ = run_gpu(wl)
    assert (h(out["slot_row"]) >= 0).all()
    np.testing.assert_array_equal(h(out["counts"]), h(out["kept"]))
    assert int(h(out["offsets"])[-1]) == wl.T * wl.k
    check_forward(wl, inp, out, e2e_tokens=64)


@pytest.mark.parametrize("name", ["bf16_t8192_d2048_e64_top6", "fp32_t512_d128_e8_top2",
                                  "decode_bf16_t64_d7168_e256_top8"])
def test_forward_with_selection_bias_and_health(name):
    # The whole layer routed with a selection-only bias, with the routing-
    # health indicators computed in the dispatch; every output against the
    # oracle routed with the same bias.
    wl = W[name]
    if wl.T > 4096:
        wl = wl.replace(T=3000)
    inp = inputs.make_inputs(wl, "cuda", expert_bias=True)
    inp["sel_bias"] = torch.randn(wl.E, generator=torch.Generator("cuda").manual_seed(3),
                                  device="cuda")
    _, inp, out, _ = run_gpu(wl, inp=inp, health=True)
    check_forward(wl, inp, out, full=wl.T <= 3000)


def test_routing_health_call_matches_oracle():
    import oracle
    rng = np.random.default_rng(8)
    for E, T, k in [(8, 4096, 2), (256, 32768, 8), (1, 5, 1), (1024, 300, 16)]:
        counts = rng.multinomial(T * k, rng.dirichlet(np.full(E, 0.3))).astype(np.int32)
        kept = np.minimum(counts, int(1.1 * T * k / E) + 1).astype(np.int32)
        wl = inputs.Workload("h", T, 64, 64, E, k, 1.0, True, "gelu_tanh", "bf16", 0, "zero")
        cfg = moe.config_from_workload(wl)
        hdev = torch.empty(4, dtype=torch.float32, device="cuda")
        moe.routing_health(cfg, torch.as_tensor(counts, device="cuda"),
                           torch.as_tensor(kept, device="cuda"), hdev)
        torch.cuda.synchronize()
        ref = oracle.routing_health(counts, kept, T, k)
        np.testing.assert_allclose(h(hdev), ref, rtol=1e-4, atol=1e-6)


REROUTE_CASES = [
    ("e64_top6", W["bf16_t8192_d2048_e64_top6"].replace(T=3000)),
    ("fp32_e8_top2", W["fp32_t512_d128_e8_top2"]),
    ("heavy_drops", inputs.Workload("heavy_drops", 700, 128, 256, 16, 4, 0.3, True, "gelu_tanh",
                                    "bf16", 21, "zipf:0.8")),
    ("decode_t64_e256", W["decode_bf16_t64_d7168_e256_top8"]),
    ("e8_top1_skewed", W["bf16_t16384_d4096_e8_top1"].replace(T=2048)),
]


@pytest.mark.parametrize("name,wl", REROUTE_CASES, ids=[c[0] for c in REROUTE_CASES])
def test_forward_with_overflow_reroute(name, wl):
    # Overflowing slots offered once to the token's next candidate, served
    # first come into the room left: every index and output against the
    # oracle's reroute fill; fewer slots are dropped than without it.
    _, inp, out, _ = run_gpu(wl, expert_bias=True, health=True, reroute=True)
    check_forward(wl, inp, out, full=wl.T <= 3000, reroute=True)
    _, _, plain, _ = run_gpu(wl, inp=inp)
    assert int(h(out["offsets"])[-1]) >= int(h(plain["offsets"])[-1])
    np.testing.assert_array_equal(h(out["counts"]), h(plain["counts"]))


def test_reroute_with_selection_bias():
    wl = W["bf16_t8192_d2048_e64_top6"].replace(T=2000, capacity_factor=0.8)
    inp = inputs.make_inputs(wl, "cuda")
    inp["sel_bias"] = inputs.selection_bias(wl, "cuda")
    _, inp, out, _ = run_gpu(wl, inp=inp, health=True, reroute=True)
    check_forward(wl, inp, out, full=True, reroute=True)


def test_bounded_wait_gives_up_and_reports_timeout():
    # A wait on a barrier that nothing signals (the same bounded wait the
    # tensor-core kernels use) must give up after its limit, record
    # MOE_ERR_TIMEOUT in the status word and leave the context usable.
    import time

    wl = W["bf16_t4096_d1024_e8_top2"]
    cfg = moe.config_from_workload(wl, write_logits=True)
    ws = moe.workspace(cfg)
    torch.cuda.synchronize()
    t0 = time.time()
    moe.selftest_wait_timeout(ws, 50_000_000)  # 50 ms
    torch.cuda.synchronize()
    assert time.time() - t0 < 5.0
    assert moe.device_status(ws) == moe.MOE_ERR_TIMEOUT
    moe.workspace_init(ws)
    torch.cuda.synchronize()
    assert moe.device_status(ws) == moe.MOE_OK
    inp = inputs.make_inputs(wl, "cuda")
    out = moe.allocate(cfg)
    moe.forward(cfg, inp, out, ws, 1.0)
    torch.cuda.synchronize()
    assert moe.device_status(ws) == moe.MOE_OK
    check_forward(wl, inp, out, n_tokens=256)


def test_grid_barrier_gives_up_and_reports_timeout():
    # The one-pass dispatch's grid barrier, waiting for one block more than
    # the grid holds, must give up after its limit and record MOE_ERR_TIMEOUT;
    # its counters return to zero, so a whole layer with a one-pass dispatch
    # (T > 256) then runs correctly on the same workspace.
    import time

    wl = W["bf16_t8192_d2048_e64_top6"].replace(T=3000)
    cfg = moe.config_from_workload(wl, write_logits=True)
    ws = moe.workspace(cfg)
    torch.cuda.synchronize()
    t0 = time.time()
    moe.selftest_grid_barrier_timeout(ws, 50_000_000)  # 50 ms
    torch.cuda.synchronize()
    assert time.time() - t0 < 5.0
    assert moe.device_status(ws) == moe.MOE_ERR_TIMEOUT
    moe.workspace_init(ws)
    torch.cuda.synchronize()
    inp = inputs.make_inputs(wl, "cuda")
    out = moe.allocate(cfg)
    moe.forward(cfg, inp, out, ws, 1.0)
    torch.cuda.synchronize()
    assert moe.device_status(ws) == moe.MOE_OK
    check_forward(wl, inp, out, n_tokens=256)


ONEPASS_CASES = [
    ("e64_top6", W["bf16_t8192_d2048_e64_top6"].replace(T=3000), False),
    ("e256_top8_ragged", W["bf16_t32768_d7168_e256_top8"].replace(T=12001, d=256, d_ff=512,
                                                                  capacity_factor=2.0), True),
    ("e8_top2_full", W["bf16_t4096_d1024_e8_top2"], False),
    ("e1024_top16", inputs.Workload("e1024", 700, 64, 64, 1024, 16, 1.0, True, "gelu_tanh",
                                    "bf16", 5, "normal:1.0"), True),
]


@pytest.mark.parametrize("name,wl,extras", ONEPASS_CASES, ids=[c[0] for c in ONEPASS_CASES])
def test_one_pass_dispatch_equals_two_kernel_dispatch(name, wl, extras):
    # With T > 256 (and no reroute) the dispatch is one cooperative grid
    # (counts, capacity, offsets and positions in one launch behind a grid
    # barrier); MOE_DISPATCH_ONEPASS=0 runs the histogram and assign kernels.
    # Every integer output, the permuted rows and the statistics (with the
    # selection bias and the routing-health outputs) must be identical.
    inp = inputs.make_inputs(wl, "cuda")
    if extras:
        inp["sel_bias"] = inputs.selection_bias(wl, "cuda")
    _, _, out1, ws1 = run_gpu(wl, inp=inp, health=extras)
    os.environ["MOE_DISPATCH_ONEPASS"] = "0"
    try:
        _, _, out2, ws2 = run_gpu(wl, inp=inp, health=extras)
    finally:
        del os.environ["MOE_DISPATCH_ONEPASS"]
    assert moe.device_status(ws1) == moe.MOE_OK and moe.device_status(ws2) == moe.MOE_OK
    names = ["counts", "kept", "offsets", "slot_row", "psum", "f", "pbar", "l_aux", "y"]
    if extras:
        names.append("health")
    for n_ in names:
        assert torch.equal(out1[n_], out2[n_]), n_
    n = int(h(out1["offsets"])[-1])
    for n_ in ["row_token", "xd"]:
        assert torch.equal(out1[n_][:n], out2[n_][:n]), n_
    check_forward(wl, inp, out1, n_tokens=256, e2e_tokens=32)

