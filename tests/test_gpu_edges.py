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
