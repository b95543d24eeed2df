"""moe_dispatch_noalloc: the dispatch stage for callers that cannot allocate
device memory of their own (for example a plugin whose host framework's
memory pool owns the whole device), so cannot hand moe_dispatch a workspace.
It keeps its scratch in a fixed array inside the library.

Checked through the C ABI against moe_dispatch (which uses a workspace) on
the same inputs, on two calls in a row, so a call that reused stale contents
of the shared array would show.  Every dispatch output is integer or an
exact row copy, so the comparison is bit-exact, as in the other dispatch
tests.  The file is named to be collected last."""

import numpy as np
import pytest
import torch

from routing_dispatch_expert_06_b300 import build, inputs, moe

pytestmark = pytest.mark.gpu

OUTPUTS = ["counts", "kept", "offsets", "slot_row"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    moe.load()


def _route(wl, seed):
    inp = inputs.make_inputs(wl, "cuda", seed=seed)
    cfg = moe.config_from_workload(wl)
    ws = moe.workspace(cfg)
    out = moe.allocate(cfg)
    moe.route(cfg, inp["x"], inp["Wr"], inp["br"], out, ws)
    return cfg, inp, out, ws


def _compare(ref, got):
    for name in OUTPUTS:
        assert torch.equal(ref[name], got[name]), name
    n = int(ref["offsets"][-1])
    assert torch.equal(ref["row_token"][:n], got["row_token"][:n])
    assert torch.equal(ref["xd"][:n], got["xd"][:n])


@pytest.mark.parametrize("name", ["bf16_t8192_d2048_e64_top6", "fp32_t512_d128_e8_top2"])
def test_noalloc_dispatch_matches_workspace_dispatch_twice(name):
    wl = inputs.WORKLOADS[name]
    # two different routings back to back: the second call must not be
    # affected by what the first left in the shared scratch array
    for seed in (wl.seed, wl.seed + 17):
        cfg, inp, ref, ws = _route(wl, seed)
        moe.dispatch(cfg, inp["x"], ref["topk_ids"], ref, ws)
        got = moe.allocate(cfg)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        moe.dispatch_noalloc(cfg, inp["x"], ref["topk_ids"], got, status)
        torch.cuda.synchronize()
        assert int(status.item()) == moe.MOE_OK
        assert moe.device_status(ws) == moe.MOE_OK
        _compare(ref, got)
        assert int(ref["offsets"][-1]) > 0


def test_noalloc_dispatch_matches_oracle():
    # Directly against the oracle's fill and permutation, on the device's
    # routing of a small layer.
    import oracle
    wl = inputs.WORKLOADS["bf16_t4096_d1024_e8_top2"].replace(T=1000, capacity_factor=0.9)
    cfg, inp, ref, ws = _route(wl, wl.seed)
    got = moe.allocate(cfg)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.dispatch_noalloc(cfg, inp["x"], ref["topk_ids"], got, status)
    torch.cuda.synchronize()
    assert int(status.item()) == moe.MOE_OK
    ids = inputs.to_numpy(ref["topk_ids"])
    fl = oracle.fill(ids, wl.E, moe.capacity(cfg))
    for name in OUTPUTS:
        np.testing.assert_array_equal(inputs.to_numpy(got[name]), fl[name], name)
    n = int(fl["offsets"][-1])
    assert 0 < n < wl.T * wl.k  # c = 0.9 drops some slots
    np.testing.assert_array_equal(inputs.to_numpy(got["row_token"])[:n], fl["row_token"])
    x = inputs.to_numpy(inp["x"])
    np.testing.assert_array_equal(inputs.to_numpy(got["xd"])[:n], x[fl["row_token"]])


def test_noalloc_fused_dispatch_matches_workspace_dispatch():
    # With fuse_dispatch no row is copied (xd is NULL); every index output
    # equals moe_dispatch's.
    wl = inputs.WORKLOADS["bf16_t8192_d2048_e64_top6"].replace(T=3000)
    inp = inputs.make_inputs(wl, "cuda")
    cfg = moe.config_from_workload(wl, fuse_dispatch=True)
    ws = moe.workspace(cfg)
    ref = moe.allocate(cfg)
    assert ref["xd"] is None
    moe.route(cfg, inp["x"], inp["Wr"], inp["br"], ref, ws)
    moe.dispatch(cfg, inp["x"], ref["topk_ids"], ref, ws)
    for _ in range(2):
        got = moe.allocate(cfg)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        moe.dispatch_noalloc(cfg, inp["x"], ref["topk_ids"], got, status)
        torch.cuda.synchronize()
        assert int(status.item()) == moe.MOE_OK
        for name in OUTPUTS:
            assert torch.equal(ref[name], got[name]), name
        n = int(ref["offsets"][-1])
        assert torch.equal(ref["row_token"][:n], got["row_token"][:n])


def test_noalloc_rejects_oversize_before_launch():
    # ceil(T/256)*E above the fixed 262144-entry scratch
    cfg = moe.config(T=1 << 20, d=64, d_ff=64, E=128, k=1, capacity_factor=1.0)
    out = {k: torch.empty(8, dtype=torch.int32, device="cuda") for k in
           ["counts", "kept", "offsets", "slot_row", "row_token"]}
    out["xd"] = torch.empty(64, dtype=torch.bfloat16, device="cuda")
    x = torch.empty(64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.dispatch_noalloc(cfg, x, out["counts"], out)
    assert ei.value.code == moe.MOE_ERR_INVALID_ARG
    assert "scratch" in str(ei.value)
