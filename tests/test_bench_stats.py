"""The bench line's load and tile figures, on hand-made cases (CPU only)."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.mark.parametrize("E,pair,kept,rows", [
    # fewer than 128 experts: whole 256-row pair tiles per expert
    (8, True, [0, 1, 256, 257], 0 + 256 + 256 + 512),
    # 128 or more experts: whole pair tiles, then a pair tile for a remainder
    # above 128 rows or a 128-row one-CTA tile for 1..128 rows
    (256, True, [1, 128, 129, 256, 300, 400], 128 + 128 + 256 + 256 + 384 + 512),
    # one CTA per tile: 128-row tiles
    (8, False, [1, 128, 129, 300], 128 + 128 + 256 + 384),
])
def test_gemm_tile_rows(E, pair, kept, rows):
    assert bench.gemm_tile_rows(kept, E, pair=pair) == rows


def test_routing_stats():
    # T = 4, k = 2, E = 2, C = 4: expert 0 is asked for 6 slots and keeps 4;
    # token 3 loses both of its slots.
    counts, kept = [6, 2], [4, 2]
    slot_row = [[0, 4], [1, 5], [2, -1], [-1, -1]]
    st = bench.routing_stats(counts, kept, slot_row, T=4, k=2, E=2, regular_gemm=True)
    assert st["dropped_slots"] == 2 and st["dropped_slot_share"] == 0.25
    assert st["overflow_tokens"] == 1
    assert st["load_max_over_mean"] == 1.5
    assert st["padding_rows"] == 0
    assert st["gemm_tile_rows"] == 512 and st["tile_waste"] == pytest.approx(512 / 6 - 1)
    st = bench.routing_stats(counts, kept, slot_row, T=4, k=2, E=2, regular_gemm=False)
    assert st["gemm_tile_rows"] is None and st["tile_waste"] is None


def test_kernel_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    # The ncu figure is reported only while the summary's recorded source hash
    # matches the kernel source; after any edit it is null.
    import hashlib

    src = tmp_path / "kernel.cu"
    src.write_text("// kernel v1\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "ffn_up_wl.md").write_text(
        f"kernel_source_sha256: {sha}\ntraffic_bytes_per_launch: 117502464\n")
    monkeypatch.setattr(bench, "PROFILES", str(prof))
    assert bench.kernel_traffic("ffn_up", "wl", str(src)) == 117502464.0
    assert bench.kernel_traffic("ffn_down", "wl", str(src)) is None  # no summary
    src.write_text("// kernel v2\n")
    assert bench.kernel_traffic("ffn_up", "wl", str(src)) is None


def test_cpu_sample_is_a_bounded_power_of_two_prefix():
    from routing_dispatch_expert_06_b300 import inputs

    W = inputs.WORKLOADS
    # the two small layers run whole; the largest layer runs a 512-token
    # prefix (474 MFLOP per token against a 3e11 budget)
    assert bench.cpu_sample_tokens(W["fp32_t512_d128_e8_top2"]) == 512
    assert bench.cpu_sample_tokens(W["bf16_t4096_d1024_e8_top2"]) == 4096
    assert bench.cpu_sample_tokens(W["bf16_t32768_d7168_e256_top8"]) == 512
    for wl in W.values():
        S = bench.cpu_sample_tokens(wl)
        assert 1 <= S <= wl.T and S & (S - 1) == 0
        per_token = 2 * wl.d * wl.E + wl.k * 4 * wl.d * wl.d_ff
        assert S == 1 or S * per_token <= 3e11
    assert inputs.DEFAULT_BENCH == "bf16_t32768_d7168_e256_top8"
