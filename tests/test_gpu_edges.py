"""Edge cases of the whole layer, through the C ABI, checked in full against
the oracle (every logit, id, index, buffer row, expert output and token).

Covered: one token; the smallest widths (d = d_ff = 8, a single 16-byte
vector per row); E = 1; the largest expert count the library accepts
(E = 1024, k = 16: the CUDA-core router, a grouped GEMM over mostly empty
experts with one-CTA tails); a capacity so small that most tokens lose every
slot (their output must be exactly 0); token counts that leave a ragged last
router tile (128) and dispatch chunk (256); d not a multiple of the 64-wide
k-block and d_ff giving an odd column tile (K tail and masked columns); the
fp32 path with many experts.
"""

import numpy as np
import pytest

from routing_dispatch_expert_06_b300 import build, inputs, moe

from parity import check_forward, h, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    moe.load()


def wl_of(name, T, d, d_ff, E, k, c, renorm=True, act="gelu_tanh", dtype="bf16",
          bias="normal:1.0", seed=21):
    return inputs.Workload(name, T, d, d_ff, E, k, c, renorm, act, dtype, seed, bias)


CASES = [
    wl_of("one_token", 1, 64, 128, 8, 2, 1.0),
    wl_of("smallest_width", 3, 8, 8, 1, 1, 1.0),
    wl_of("max_experts_top16", 300, 64, 64, 1024, 16, 1.0),
    wl_of("almost_all_dropped", 700, 128, 256, 16, 4, 0.05),
    wl_of("ragged_tiles", 257, 136, 200, 24, 3, 1.3, renorm=False),
    wl_of("k_tail_odd_bn", 1000, 72, 136, 8, 2, 1.25),
    wl_of("wide_experts_256", 1000, 256, 256, 256, 8, 1.25, renorm=False),
    wl_of("fp32_many_experts", 400, 64, 96, 300, 5, 1.0, act="relu", dtype="f32"),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_edge_case_matches_oracle(wl):
    _, inp, out, _ = run_gpu(wl, expert_bias=True)
    info = check_forward(wl, inp, out, full=True)
    assert info["n_rows"] <= wl.T * wl.k


def test_fully_dropped_tokens_output_zero():
    wl = CASES[3]
    _, inp, out, _ = run_gpu(wl)
    slot = h(out["slot_row"])
    dropped = (slot < 0).all(axis=1)
    assert dropped.sum() > wl.T // 2  # the tiny capacity drops most tokens entirely
    y = inputs.as_f64(h(out["y"]))
    assert (y[dropped] == 0).all()


# ---- caller-supplied expert ids: repeats within a token, ids out of range ----

def _ids_case(T, E, k, seed):
    """Host-built ids: a random distinct set per token, as a router gives."""
    rng = np.random.default_rng(seed)
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32), rng


def _dispatch_with(cfg, x, ids_host, noalloc=False):
    import torch
    ids = torch.as_tensor(ids_host, device="cuda")
    out = moe.allocate(cfg)
    ws = moe.workspace(cfg)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if noalloc:
        moe.dispatch_noalloc(cfg, x, ids, out, status)
    else:
        moe.dispatch(cfg, x, ids, out, ws)
    torch.cuda.synchronize()
    st = int(status.item()) if noalloc else moe.device_status(ws)
    return out, st


@pytest.mark.parametrize("noalloc", [False, True], ids=["workspace", "noalloc"])
def test_repeated_expert_within_a_token_matches_oracle_fill(noalloc):
    # Every (t, r) is its own slot; two ranks of one token naming the same
    # expert take consecutive positions in rank order, exactly as the
    # oracle's sequential fill gives them.
    import oracle
    T, E, k = 700, 8, 4
    wl = wl_of("repeats", T, 64, 64, E, k, 1.0)
    cfg = moe.config_from_workload(wl)
    ids, rng = _ids_case(T, E, k, 5)
    rep = rng.random(T) < 0.3
    ids[rep, 2] = ids[rep, 0]          # rank 2 repeats rank 0
    ids[rep[::-1], 3] = ids[rep[::-1], 1]
    x = inputs.make_inputs(wl, "cuda")["x"]
    out, st = _dispatch_with(cfg, x, ids, noalloc)
    assert st == moe.MOE_OK
    fl = oracle.fill(ids, E, moe.capacity(cfg))
    for name in ["counts", "kept", "offsets", "slot_row"]:
        np.testing.assert_array_equal(h(out[name]), fl[name], name)
    n = int(fl["offsets"][E])
    np.testing.assert_array_equal(h(out["row_token"])[:n], fl["row_token"])
    np.testing.assert_array_equal(h(out["xd"])[:n], h(x)[fl["row_token"]])


@pytest.mark.parametrize("noalloc", [False, True], ids=["workspace", "noalloc"])
def test_out_of_range_ids_are_skipped_and_reported(noalloc):
    # An id outside [0, E) names no expert: its slot is not counted, its
    # slot_row is -1, the status word says MOE_ERR_INVALID_ARG, and every
    # other slot is dispatched as if that slot were absent.  Expected values:
    # the oracle's fill with the bad slots sent to an extra expert E placed
    # after all real ones (same capacity C), which leaves experts 0..E-1,
    # their rows and their offsets exactly as without those slots.
    import oracle
    T, E, k = 512, 8, 2
    wl = wl_of("bad_ids", T, 64, 64, E, k, 1.0)
    cfg = moe.config_from_workload(wl)
    ids, rng = _ids_case(T, E, k, 6)
    bad = rng.random((T, k)) < 0.05
    ids[bad] = np.where(rng.random(bad.sum()) < 0.5, E, -3)
    x = inputs.make_inputs(wl, "cuda")["x"]
    out, st = _dispatch_with(cfg, x, ids, noalloc)
    assert st == moe.MOE_ERR_INVALID_ARG
    C = moe.capacity(cfg)
    fl = oracle.fill(np.where(bad, E, ids).astype(np.int32), E + 1, C)
    np.testing.assert_array_equal(h(out["counts"]), fl["counts"][:E])
    np.testing.assert_array_equal(h(out["kept"]), fl["kept"][:E])
    np.testing.assert_array_equal(h(out["offsets"]), fl["offsets"][:E + 1])
    want = np.where(bad, -1, fl["slot_row"])
    np.testing.assert_array_equal(h(out["slot_row"]), want)
    n = int(fl["offsets"][E])
    np.testing.assert_array_equal(h(out["row_token"])[:n], fl["row_token"][:n])
    np.testing.assert_array_equal(h(out["xd"])[:n], h(x)[fl["row_token"][:n]])
