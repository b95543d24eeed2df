"""Benchmark: forward pass of one MoE layer on B300, tokens/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline]

One step = one forward pass of the whole layer (route, dispatch, grouped
expert FFN, combine, aux statistics) over one batch of T synthetic tokens,
inputs already resident in HBM.  The pass (one moe_forward call) is captured
once into a CUDA graph and each step replays it, timed with CUDA events on
the stream, with the L2 cache flushed between steps outside the events (a
512 MiB write, then a 512 MiB read so that the write's dirty lines are
written back before the timed step).  Per-stage times come from one graph per stage, replayed the
same way; the eager time of moe_forward launched from Python is reported
beside them.  Rank 0 prints one JSON line.

Multi-GPU: the layer does not shard in this design (replicas only), so under
torchrun every rank runs an independent replica on its own batch and
``value`` is the tokens of all ranks / the slowest rank's time.

``--impl reference`` times the CPU oracle (the plain C++ implementation the
tests compare against) on the host cores, W untimed and K timed forward passes
over a bounded sample of the same workload (its first S tokens as one layer
call, S from cpu_sample_tokens), and prints the same JSON line with
"impl": "reference".  The GPU arm's cpu_baseline times the same sample.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import torch

from routing_dispatch_expert_06_b300 import inputs

ROOT = os.path.dirname(os.path.abspath(__file__))
PROFILES = os.path.join(ROOT, "profiles")
STAGES = ["route", "dispatch", "ffn_up", "ffn_down", "combine", "aux"]
METRIC = "MoE-layer fwd tokens/s on 1 B300; grouped-FFN TC util %; dispatch HBM GB/s"


# ---------------------------------------------------------------- helpers ----

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6400.0, bf16=1800.0, bf16_sustained=1400.0, source="fallback")


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[3:]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return dict(sm_mhz=statistics.median(sm), sm_max_mhz=max(mx), reasons=sorted(reasons),
                    samples=len(sm))


def kernel_traffic(kernel: str, workload: str, src_file: str):
    """DRAM bytes per launch from the committed ncu summary, if it still
    describes the current kernel source (sha256 match), else None."""
    path = os.path.join(PROFILES, f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_h = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", text)
    if not (m_t and m_h):
        return None
    with open(src_file, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != m_h.group(1):
            return None
    return float(m_t.group(1))


def algorithmic(wl, n_kept: int, t_kept: int, fused: bool = False):
    """Bytes / FLOPs the method must move or compute per forward pass
    (``fused``: the dispatch moves no rows, only ids, positions and
    row_token; the first GEMM reads the token rows itself)."""
    b = 2 if wl.dtype == "bf16" else 4
    T, d, d_ff, E, k = wl.T, wl.d, wl.d_ff, wl.E, wl.k
    rows = 0 if fused else t_kept * d * b + n_kept * d * b
    return dict(
        route_bytes=T * d * b + E * d * b + T * k * 8,
        route_flops=2 * T * d * E,
        dispatch_bytes=rows + T * k * 8 + n_kept * 4,
        ffn_up_flops=2 * n_kept * d * d_ff,
        ffn_down_flops=2 * n_kept * d * d_ff,
        combine_bytes=n_kept * d * b + T * k * 8 + T * d * b,
    )


def gemm_tile_rows(kept, E: int, pair: bool = True, tail_split_min_experts: int = 128) -> int:
    """Rows the regular tensor-core grouped GEMM computes for experts holding
    ``kept`` rows: tiles never straddle two experts, so each expert's rows are
    rounded up to whole tiles (256 rows for a CTA pair, 128 for one CTA; with
    E >= 128 an expert's last 1..128 rows go to one 128-row tile)."""
    total = 0
    for r in (int(v) for v in kept):
        if r <= 0:
            continue
        if not pair:
            total += -(-r // 128) * 128
        elif E >= tail_split_min_experts:
            whole, rem = divmod(r, 256)
            total += whole * 256 + (256 if rem > 128 else 128 if rem > 0 else 0)
        else:
            total += -(-r // 256) * 256
    return total


def routing_stats(counts, kept, slot_row, T: int, k: int, E: int, regular_gemm: bool):
    """Load and drop figures of one forward pass (the monitoring list of
    [MoE 模型原理 §4.4] and the evaluation list of §13): slots dropped by
    the capacity, tokens with no kept slot, the hottest expert's load over the
    mean, the dispatch buffer's padding (none: it is ragged) and the regular
    GEMM's tile waste (rows computed in partial tiles over kept rows; None
    for the swapped decode GEMM and the CUDA-core GEMM, tiled otherwise)."""
    counts = [int(v) for v in counts]
    kept = [int(v) for v in kept]
    n_kept = sum(kept)
    t_kept = sum(1 for row in slot_row if any(int(v) >= 0 for v in row))
    tile_rows = gemm_tile_rows(kept, E) if regular_gemm else None
    return dict(
        dropped_slots=T * k - n_kept,
        dropped_slot_share=(T * k - n_kept) / (T * k),
        overflow_tokens=T - t_kept,
        load_max_over_mean=max(counts) * E / (T * k),
        padding_rows=0,
        gemm_tile_rows=tile_rows,
        tile_waste=(tile_rows / n_kept - 1.0) if (tile_rows is not None and n_kept) else None,
    )


# ------------------------------------------------------------ CPU oracle ----

def cpu_model() -> str:
    """The host CPU's model name (from /proc/cpuinfo), or '' if unknown."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return ""


def cpu_sample_tokens(wl, flop_budget: float = 3e11) -> int:
    """Tokens S of the CPU oracle's timed sample: the largest power of two,
    at most T, whose forward pass costs at most ``flop_budget`` of the
    method's arithmetic (router 2·d·E plus expert FFN k·4·d·d_ff per token),
    i.e. a few seconds of the oracle on a host's cores."""
    per_token = 2 * wl.d * wl.E + wl.k * 4 * wl.d * wl.d_ff
    S = 1
    while S * 2 <= wl.T and S * 2 * per_token <= flop_budget:
        S *= 2
    return S


def sample_text(wl, S: int) -> str:
    return (f"the first {S} of the {wl.T} tokens of the {wl.name} batch (same seeded x and "
            f"weights as the GPU run), routed and computed as one layer call of the C++ "
            f"oracle (capacity over the {S} tokens)")


def host_inputs(wl, inp, S: int):
    """Host copies (numpy; bf16 as uint16 bits) of the workload's tensors,
    with x cut to its first S tokens."""
    out = {k: inputs.to_numpy(v) for k, v in inp.items() if k not in ("x", "sel_bias")}
    out["x"] = inputs.to_numpy(inp["x"][:S])
    return out


def oracle_forward_seconds(wl, host) -> float:
    """Wall time of one oracle forward pass over host["x"] (its own capacity
    group)."""
    import oracle  # test infrastructure: only the CPU-baseline legs run it

    act = oracle.ACT_RELU if wl.act == "relu" else oracle.ACT_GELU_TANH
    t0 = time.perf_counter()
    oracle.forward(host["x"], host["Wr"], host["br"], host["W1"], host["b1"], host["W2"],
                   host["b2"], k=wl.k, capacity_factor=wl.capacity_factor,
                   renormalize=wl.renormalize, act=act)
    return time.perf_counter() - t0


def cpu_oracle_sample(wl, inp):
    """The oracle timed on the host cores on the bounded sample of this
    workload (one untimed run, then one timed run).  Returns the bench line's
    cpu_baseline object (tokens/s of the sample)."""
    import oracle

    S = cpu_sample_tokens(wl)
    host = host_inputs(wl, inp, S)
    oracle_forward_seconds(wl, host)
    dt = oracle_forward_seconds(wl, host)
    return dict(value=S / dt, unit="tokens/s", cores=oracle.num_threads(), kind="oracle",
                cpu_model=cpu_model(), sample=f"{sample_text(wl, S)}; {dt:.2f} s")


def max_over_ranks(value, dist=None, device=None):
    """The slowest rank's value (an all-reduce MAX over the process group;
    the value itself without one)."""
    t = torch.tensor([float(value)], dtype=torch.float64)
    if dist is not None:
        if device is not None:
            t = t.to(device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, tokens_per_rank, steps, max_ms):
    """Whole-job throughput of independent replicas: the tokens of all ranks
    over the slowest rank's time for the timed steps."""
    return world * tokens_per_rank * steps / (max_ms * 1e-3)


def replica_seed(seed, rank):
    """Seed of rank `rank`'s own batch (every replica routes different tokens)."""
    return seed * 1000 + rank


def bench_config(wl, args, world):
    """The line's config object (the same on both arms)."""
    return dict(workload=wl.name, T=wl.T, d=wl.d, d_ff=wl.d_ff, E=wl.E, k=wl.k,
                capacity_factor=wl.capacity_factor, renormalize=wl.renormalize, act=wl.act,
                parallelism=f"replicas{world}" if world > 1 else "single",
                sel_bias=bool(args.sel_bias), health=bool(args.health),
                reroute=bool(args.reroute), fuse_dispatch=bool(args.fuse_dispatch),
                fuse_combine=bool(args.fuse_combine),
                l2="flushed between steps (512 MiB write, then 512 MiB read)")


def run_reference(args, wl, rank, world):
    """The oracle arm: W untimed and K timed forward passes of the C++ oracle
    on the host cores, each over the same bounded sample the GPU arm's
    cpu_baseline uses (cpu_sample_tokens), inputs drawn by the same seeded
    recipe (on the GPU when there is one, so the bytes are the GPU arm's).
    ms_per_step is the measured mean seconds of one such forward."""
    if rank != 0:
        return 0
    import oracle

    S = cpu_sample_tokens(wl)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = inputs.make_inputs(wl, dev)
    host = host_inputs(wl, inp, S)
    del inp
    for _ in range(args.warmup):
        oracle_forward_seconds(wl, host)
    times = [oracle_forward_seconds(wl, host) for _ in range(args.steps)]
    total = sum(times)
    v = S * len(times) / total
    cfg = bench_config(wl, args, world)
    cfg["l2"] = "n/a (CPU)"
    line = dict(metric=METRIC, value=v, unit="tokens/s", n_gpus=world, steps=len(times),
                warmup=args.warmup, ms_per_step=1e3 * total / len(times), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic", config=cfg,
                impl="reference",
                cpu_baseline=dict(value=v, unit="tokens/s", cores=oracle.num_threads(),
                                  kind="oracle", cpu_model=cpu_model(),
                                  sample=f"{sample_text(wl, S)}; each step one forward of it"),
                e2e=dict(value=v, unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- GPU bench ----

def capture(fn):
    """Capture the launches of fn() into a CUDA graph (on torch's capture
    stream, which the library calls pick up as the current stream)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=inputs.DEFAULT_BENCH, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--alpha", type=float, default=0.01)
    ap.add_argument("--sel-bias", action="store_true",
                    help="route with a seeded selection-only expert bias")
    ap.add_argument("--health", action="store_true",
                    help="also compute the routing-health indicators in the forward pass")
    ap.add_argument("--reroute", action="store_true",
                    help="offer overflowing slots to the token's next candidate")
    ap.add_argument("--fuse-dispatch", action="store_true",
                    help="no dispatch buffer: the first GEMM gathers the token rows")
    ap.add_argument("--fuse-combine", action="store_true",
                    help="the second GEMM also combines (no separate combine launch)")
    args = ap.parse_args()
    wl = inputs.WORKLOADS[args.workload]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, wl, rank, world)

    from routing_dispatch_expert_06_b300 import build, moe

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if rank == 0:
        build.build()
    if dist is not None:
        dist.barrier()
    moe.load()

    dev = torch.device("cuda", local_rank)
    inp = inputs.make_inputs(wl, dev)
    if args.sel_bias:
        inp["sel_bias"] = inputs.selection_bias(wl, dev)
    if world > 1:  # each replica routes its own batch
        g = torch.Generator(device=dev).manual_seed(replica_seed(wl.seed, rank))
        inp["x"] = torch.randn(inp["x"].shape, generator=g, device=dev).to(inp["x"].dtype)
    cfg = moe.config_from_workload(wl, write_logits=False, reroute=args.reroute,
                                   fuse_dispatch=args.fuse_dispatch,
                                   fuse_combine=args.fuse_combine)
    ws = moe.workspace(cfg, dev)
    out = moe.allocate(cfg, dev, health=args.health)
    stream = torch.cuda.current_stream(dev)
    flush_w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(512 << 20, dtype=torch.uint8, device=dev)

    def flush_l2():
        # Evict L2 between steps, outside the timed events: write a buffer
        # larger than L2, then read another one, so the write's dirty lines
        # are written back here instead of by the first timed kernel.
        flush_w.zero_()
        flush_r.sum(dtype=torch.int32)

    for _ in range(max(args.warmup, 3)):
        moe.forward_stages(cfg, inp, out, ws, args.alpha, stream)
    torch.cuda.synchronize(dev)

    # The forward pass is captured once into a CUDA graph (every library call
    # only enqueues kernels), as a serving loop would run it; each timed step
    # replays it.  Per-stage times come from one graph per stage.
    launches0 = moe.launch_count()
    g_full = capture(lambda: moe.forward(cfg, inp, out, ws, args.alpha))
    per_forward = moe.launch_count() - launches0
    stage_calls = {
        "route": lambda: moe.route(cfg, inp["x"], inp["Wr"], inp["br"], out, ws,
                                   sel_bias=inp.get("sel_bias")),
        "dispatch": lambda: moe.dispatch(cfg, inp["x"], out["topk_ids"], out, ws),
        "ffn_up": (lambda: moe.ffn_up_gather(cfg, inp["x"], out["row_token"], out["offsets"],
                                             inp["W1"], inp["b1"], out["H"], ws))
        if args.fuse_dispatch else
        (lambda: moe.ffn_up(cfg, out["xd"], out["offsets"], inp["W1"], inp["b1"], out["H"], ws)),
        "ffn_down": (lambda: moe.ffn_down_combine(cfg, out["H"], out["offsets"],
                                                  out["row_token"], out["slot_row"],
                                                  out["topk_w"], inp["W2"], inp["b2"], out["yd"],
                                                  out["y"], ws))
        if args.fuse_combine else
        (lambda: moe.ffn_down(cfg, out["H"], out["offsets"], inp["W2"], inp["b2"], out["yd"],
                              ws)),
        "combine": None if args.fuse_combine else
        (lambda: moe.combine(cfg, out["yd"], out["slot_row"], out["topk_w"], out["y"])),
        "aux": lambda: moe.aux_stats(cfg, out["counts"], out["psum"], args.alpha, out["f"],
                                     out["pbar"], out["l_aux"]),
    }
    # (with the combine fused into ffn_down there is no combine stage: 0 ms)
    g_stage = {name: capture(fn) for name, fn in stage_calls.items() if fn is not None}
    for _ in range(2):
        g_full.replay()
        for name in STAGES:
            if name in g_stage:
                g_stage[name].replay()
    torch.cuda.synchronize(dev)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    K = args.steps
    evs = [(ev(), ev()) for _ in range(K)]
    sevs = [[ev() for _ in range(7)] for _ in range(K)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        for s_ in range(K):
            flush_l2()
            evs[s_][0].record(stream)
            g_full.replay()
            evs[s_][1].record(stream)
        torch.cuda.synchronize(dev)
    launches = K * per_forward
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    # Stage breakdown: the same steps, one graph per stage.
    for s_ in range(K):
        flush_l2()
        for i, name in enumerate(STAGES):
            sevs[s_][i].record(stream)
            if name in g_stage:
                g_stage[name].replay()
        sevs[s_][6].record(stream)
    torch.cuda.synchronize(dev)
    # Eager reference: moe_forward launched from Python each step.
    eager_ms = 0.0
    for s_ in range(K):
        flush_l2()
        a, b = ev(), ev()
        a.record(stream)
        moe.forward(cfg, inp, out, ws, args.alpha, stream)
        b.record(stream)
        torch.cuda.synchronize(dev)
        eager_ms += a.elapsed_time(b)
    eager_ms /= K
    assert moe.device_status(ws) == moe.MOE_OK

    stage_ms = {name: 0.0 for name in STAGES}
    total_ms = 0.0
    for s_ in range(K):
        total_ms += evs[s_][0].elapsed_time(evs[s_][1])
        for i, name in enumerate(STAGES):
            stage_ms[name] += sevs[s_][i].elapsed_time(sevs[s_][i + 1])
    max_ms = max_over_ranks(total_ms, dist, dev)

    offsets = out["offsets"].cpu()
    n_kept = int(offsets[-1])
    touched = int((out["kept"].cpu() > 0).sum())
    slot = out["slot_row"].cpu()
    t_kept = int((slot >= 0).any(dim=1).sum())
    alg = algorithmic(wl, n_kept, t_kept, fused=args.fuse_dispatch)
    C = moe.capacity(cfg)
    regular_gemm = wl.dtype == "bf16" and min(C, wl.T * wl.k) > 64
    routing = routing_stats(out["counts"].cpu().tolist(), out["kept"].cpu().tolist(),
                            slot.tolist(), wl.T, wl.k, wl.E, regular_gemm)
    peaks = load_peaks()
    mean = {k: v / K for k, v in stage_ms.items()}
    ffn_ms = mean["ffn_up"] + mean["ffn_down"]
    dom = "ffn_up" if mean["ffn_up"] >= mean["ffn_down"] else "ffn_down"
    dom_tflops = alg[f"{dom}_flops"] / (mean[dom] * 1e-3) / 1e12
    dom_kernel = ("ffn_up_gather" if (dom == "ffn_up" and args.fuse_dispatch) else
                  "ffn_down_combine" if (dom == "ffn_down" and args.fuse_combine) else dom)
    traffic = kernel_traffic(dom_kernel, wl.name, os.path.join(
        ROOT, "routing_dispatch_expert_06_b300", "csrc", "ffn_tc.cu"))

    # e2e: the public call with host buffers, H2D of x and D2H of y inside
    x_host = inp["x"].cpu().pin_memory()
    y_host = torch.empty(out["y"].shape, dtype=out["y"].dtype).pin_memory()
    l_host = torch.empty(1, dtype=torch.float32).pin_memory()
    x_dev = inp["x"]
    inp_e2e = dict(inp)
    e2e_steps = max(3, min(K, 10))
    for _ in range(2):
        x_dev.copy_(x_host, non_blocking=True)
        moe.forward(cfg, inp_e2e, out, ws, args.alpha, stream)
        y_host.copy_(out["y"], non_blocking=True)
    torch.cuda.synchronize(dev)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e2e_ms = 0.0
    for _ in range(e2e_steps):
        flush_l2()
        e_start.record(stream)
        x_dev.copy_(x_host, non_blocking=True)
        moe.forward(cfg, inp_e2e, out, ws, args.alpha, stream)
        y_host.copy_(out["y"], non_blocking=True)
        l_host.copy_(out["l_aux"], non_blocking=True)
        e_end.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms += e_start.elapsed_time(e_end)
    e2e_ms /= e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    value = job_tokens_per_s(world, wl.T, K, max_ms)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(wl, inp)
    b = 2 if wl.dtype == "bf16" else 4
    hbm = peaks["hbm"]
    stage_gbs = dict(route=alg["route_bytes"] / (mean["route"] * 1e-3) / 1e9,
                     dispatch=alg["dispatch_bytes"] / (mean["dispatch"] * 1e-3) / 1e9)
    if not args.fuse_combine:  # fused: the combine's bytes move inside ffn_down
        stage_gbs["combine"] = alg["combine_bytes"] / (mean["combine"] * 1e-3) / 1e9
    ffn_tflops = alg["ffn_up_flops"] * 2 / (ffn_ms * 1e-3) / 1e12
    line = dict(
        metric=METRIC, value=value, unit="tokens/s", n_gpus=world, steps=K, warmup=args.warmup,
        ms_per_step=max_ms / K, higher_is_better=True, scaling="weak", vs_baseline=None,
        dtype="bf16" if wl.dtype == "bf16" else "f32", data="synthetic",
        config=bench_config(wl, args, world),
        roofline=dict(bound="tensor", kernel=f"{dom_kernel} (tcgen05 grouped GEMM"
                      + (", pair-body and tail launches" if wl.E >= 128 else "") + ")",
                      achieved=dom_tflops, peak=peaks["bf16"], unit="TFLOP/s",
                      frac=dom_tflops / peaks["bf16"], traffic=traffic,
                      peak_source=f"{peaks['source']} bf16 burst",
                      peak_sustained=peaks["bf16_sustained"],
                      frac_sustained=dom_tflops / peaks["bf16_sustained"]),
        cpu_baseline=cpu,
        e2e=dict(value=world * wl.T / (e2e_ms * 1e-3), unit="tokens/s",
                 h2d_bytes_per_step=wl.T * wl.d * b, d2h_bytes_per_step=wl.T * wl.d * b + 4),
        gpu_launches=launches,
        clocks=clocks.summary(),
        timing="forward captured once as a CUDA graph, replayed per step; stages_ms from "
               "one graph per stage; eager_ms_per_step = moe_forward launched from Python",
        eager_ms_per_step=eager_ms,
        stages_ms={k: round(v, 5) for k, v in mean.items()},
        ffn_tflops=ffn_tflops,
        ffn_tc_frac=ffn_tflops / peaks["bf16"],
        ffn_tc_frac_sustained=ffn_tflops / peaks["bf16_sustained"],
        dispatch_gbs=stage_gbs["dispatch"],
        combine_gbs=stage_gbs.get("combine"),
        route_gbs=stage_gbs["route"],
        hbm_peak_gbs=hbm,
        hbm_frac={k: v / hbm for k, v in stage_gbs.items()},
        kept_rows=n_kept,
        experts_touched=touched,
        routing=routing,
        # With few rows per expert the grouped FFN is bound by reading the
        # touched experts' W1 and W2: their bytes over the FFN time.
        ffn_weight_gbs=touched * 2 * wl.d * wl.d_ff * b / (ffn_ms * 1e-3) / 1e9,
    )
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
