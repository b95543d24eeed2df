"""Seeded synthetic inputs for the MoE-layer forward.

This module only draws random tensors; it holds none of the layer's
arithmetic.  Both the CUDA path (tests, benchmark) and the CPU oracle (tests,
CPU baseline) take their inputs from here, so both sides see identical bytes.

Recipe (all draws from one ``torch.Generator`` seeded per workload, in the
fixed order x, W_r, b_r, W1, b1, W2, b2; each drawn in fp32, then rounded to
bf16 with round-to-nearest-even where the workload is bf16):

* x ~ N(0, 1)
* W_r, W1, W2 ~ N(0, 1/fan_in)  (fan_in = d for W_r and W1, d_ff for W2)
* expert biases b1, b2 are 0 unless ``expert_bias`` is set (then N(0, 0.1²))
* router bias b_r per workload: a linear skew, zero, a normal draw, or a
  Zipf-like log decay — chosen so that some experts overflow their capacity.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    d_ff: int
    E: int
    k: int
    capacity_factor: float
    renormalize: bool
    act: str            # "relu" or "gelu_tanh"
    dtype: str          # "f32" or "bf16" for x and weights
    seed: int
    router_bias: str    # "linear_skew", "zero", "normal:<std>", "zipf:<a>"

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("fp32_t512_d128_e8_top2", 512, 128, 512, 8, 2, 1.0, True, "relu", "f32", 0,
                 "linear_skew"),
        Workload("bf16_t4096_d1024_e8_top2", 4096, 1024, 4096, 8, 2, 1.25, True, "gelu_tanh",
                 "bf16", 1, "zero"),
        Workload("bf16_t16384_d4096_e8_top1", 16384, 4096, 14336, 8, 1, 1.0, True, "gelu_tanh",
                 "bf16", 2, "normal:0.7071067811865476"),
        Workload("bf16_t8192_d2048_e64_top6", 8192, 2048, 1408, 64, 6, 1.0, True, "gelu_tanh",
                 "bf16", 3, "zipf:0.8"),
        Workload("bf16_t32768_d7168_e256_top8", 32768, 7168, 2048, 256, 8, 1.25, False,
                 "gelu_tanh", "bf16", 4, "normal:1.0"),
        # Decode regime: T = 1, 8, 64 tokens per call on the two many-expert
        # layers; the expert FFN is then bound by reading the touched experts'
        # weights.
        Workload("decode_bf16_t1_d7168_e256_top8", 1, 7168, 2048, 256, 8, 1.25, False,
                 "gelu_tanh", "bf16", 9, "normal:1.0"),
        Workload("decode_bf16_t8_d7168_e256_top8", 8, 7168, 2048, 256, 8, 1.25, False,
                 "gelu_tanh", "bf16", 6, "normal:1.0"),
        Workload("decode_bf16_t64_d7168_e256_top8", 64, 7168, 2048, 256, 8, 1.25, False,
                 "gelu_tanh", "bf16", 10, "normal:1.0"),
        Workload("decode_bf16_t1_d2048_e64_top6", 1, 2048, 1408, 64, 6, 1.0, True,
                 "gelu_tanh", "bf16", 11, "zipf:0.8"),
        Workload("decode_bf16_t8_d2048_e64_top6", 8, 2048, 1408, 64, 6, 1.0, True,
                 "gelu_tanh", "bf16", 12, "zipf:0.8"),
        Workload("decode_bf16_t64_d2048_e64_top6", 64, 2048, 1408, 64, 6, 1.0, True,
                 "gelu_tanh", "bf16", 7, "zipf:0.8"),
        # The largest layer's shapes (d = 7168, d_ff = 2048, top-8, N(0, 1)
        # router bias) at 1/8 of its tokens and experts: the same capacity
        # C = 1280 per expert, so the same per-expert row counts, on a few GB
        # of device memory (for hardware-counter captures of its kernels).
        Workload("bf16_t4096_d7168_e32_top8", 4096, 7168, 2048, 32, 8, 1.25, False,
                 "gelu_tanh", "bf16", 13, "normal:1.0"),
        # The largest layer's routing, dispatch and combine at full size (T =
        # 32768, d = 7168, E = 256, top-8, same seed and router) with a
        # narrow expert width d_ff = 64, so that the whole layer holds about
        # 4 GB of device memory (for hardware-counter captures of those
        # kernels; the expert GEMMs are not representative here).
        Workload("narrow_bf16_t32768_d7168_e256_top8", 32768, 7168, 64, 256, 8, 1.25, False,
                 "gelu_tanh", "bf16", 4, "normal:1.0"),
        # Dropless: c = E/k makes C = ceil(c·T·k/E) = T, so no expert can
        # overflow (every slot is kept).
        Workload("dropless_bf16_t8192_d2048_e64_top6", 8192, 2048, 1408, 64, 6, 64 / 6, True,
                 "gelu_tanh", "bf16", 8, "zipf:0.8"),
    ]
}

# Workload timed by default in the benchmark: the largest layer (T = 32768,
# d = 7168, d_ff = 2048, E = 256, top-8).
DEFAULT_BENCH = "bf16_t32768_d7168_e256_top8"


def _router_bias(kind: str, E: int, gen: torch.Generator, device) -> torch.Tensor:
    if kind == "zero":
        return torch.zeros(E, dtype=torch.float32, device=device)
    if kind == "linear_skew":
        i = torch.arange(E, dtype=torch.float64)
        return (0.5 * (E - 1 - i) / E).to(torch.float32).to(device)
    if kind.startswith("normal:"):
        std = float(kind.split(":")[1])
        return torch.randn(E, generator=gen, device=device, dtype=torch.float32) * std
    if kind.startswith("zipf:"):
        a = float(kind.split(":")[1])
        i = torch.arange(E, dtype=torch.float64)
        return (-a * torch.log(i + 1.0)).to(torch.float32).to(device)
    raise ValueError(kind)


def make_inputs(wl: Workload, device="cpu", expert_bias: bool = False, seed: int | None = None):
    """Draw x, W_r, b_r, W1, b1, W2, b2 for a workload on ``device``.

    Shapes: x [T,d]; Wr [E,d]; br [E] fp32; W1 [E,d_ff,d]; b1 [E,d_ff] fp32;
    W2 [E,d,d_ff]; b2 [E,d] fp32.  x and the weights are fp32 or bf16.
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed if seed is None else seed)
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    T, d, d_ff, E = wl.T, wl.d, wl.d_ff, wl.E

    def normal(shape, std):
        return (torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std).to(dt)

    x = normal((T, d), 1.0)
    Wr = normal((E, d), 1.0 / math.sqrt(d))
    br = _router_bias(wl.router_bias, E, gen, device)
    W1 = torch.empty((E, d_ff, d), dtype=dt, device=device)
    for e in range(E):  # one expert at a time keeps the fp32 temporaries small
        W1[e] = normal((d_ff, d), 1.0 / math.sqrt(d))
    b1 = (torch.randn((E, d_ff), generator=gen, device=device) * 0.1 if expert_bias
          else torch.zeros((E, d_ff), device=device)).to(torch.float32)
    W2 = torch.empty((E, d, d_ff), dtype=dt, device=device)
    for e in range(E):
        W2[e] = normal((d, d_ff), 1.0 / math.sqrt(d_ff))
    b2 = (torch.randn((E, d), generator=gen, device=device) * 0.1 if expert_bias
          else torch.zeros((E, d), device=device)).to(torch.float32)
    return dict(x=x, Wr=Wr, br=br, W1=W1, b1=b1, W2=W2, b2=b2)


def selection_bias(wl: Workload, device="cpu") -> torch.Tensor:
    """A seeded per-expert selection bias, N(0, 1) fp32 [E] (seed: the
    workload's + 7919), for routing with a selection-only bias."""
    gen = torch.Generator(device=torch.device(device))
    gen.manual_seed(wl.seed + 7919)
    return torch.randn(wl.E, generator=gen, device=device, dtype=torch.float32)


def to_numpy(t: torch.Tensor) -> np.ndarray:
    """Host copy; bf16 becomes a uint16 array of the same bit patterns."""
    t = t.detach().contiguous()
    if t.dtype == torch.bfloat16:
        return t.cpu().view(torch.int16).numpy().view(np.uint16)
    return t.cpu().numpy()


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Widen a uint16 array of bf16 bit patterns to float64 (exact)."""
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def as_f64(a: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)
