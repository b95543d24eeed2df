"""Python binding of libmoe.so (argument marshalling only).

Every step of the layer runs in the library's CUDA kernels; this module turns
torch tensors (device memory) and the current torch CUDA stream into the C
ABI's plain pointers and checks the returned status.  There is no fallback:
if libmoe.so is missing or cannot load, every call raises.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_WORKSPACE, \
    MOE_ERR_TIMEOUT = range(6)
MOE_DT_F32, MOE_DT_BF16 = 0, 1
MOE_ACT_RELU, MOE_ACT_GELU_TANH = 0, 1

_P = ctypes.c_void_p


class MoeError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{_status_name(code)}: {msg}")
        self.code = code


class Config(ctypes.Structure):
    """Mirror of moe_config_t."""
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("capacity_factor", ctypes.c_double), ("renormalize", ctypes.c_int32),
                ("act", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("write_logits", ctypes.c_int32), ("reroute", ctypes.c_int32),
                ("fuse_dispatch", ctypes.c_int32), ("fuse_combine", ctypes.c_int32)]


_TENSOR_FIELDS = ["x", "Wr", "br", "W1", "b1", "W2", "b2", "logits", "topk_ids", "topk_w",
                  "psum", "counts", "kept", "offsets", "slot_row", "row_token", "xd", "H", "yd",
                  "y", "f", "pbar", "l_aux", "sel_bias", "health"]


class Tensors(ctypes.Structure):
    """Mirror of moe_tensors_t (device pointers)."""
    _fields_ = [(n, _P) for n in _TENSOR_FIELDS]


_lib = None


def load():
    """Load libmoe.so (raises if it is missing: the CUDA path is the only path)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing; build it with "
                           "`python -m routing_dispatch_expert_06_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    st, i64, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    cfgp = ctypes.POINTER(Config)
    sig = {
        "moe_capacity": (i64, [cfgp]),
        "moe_max_rows": (i64, [cfgp]),
        "moe_workspace_size": (st, [cfgp, ctypes.POINTER(sz)]),
        "moe_workspace_init": (st, [_P, sz, _P]),
        "moe_route": (st, [cfgp, _P, _P, _P, _P, _P, _P, _P, _P, sz, _P]),
        "moe_route_sel": (st, [cfgp, _P, _P, _P, _P, _P, _P, _P, _P, _P, sz, _P]),
        "moe_routing_health": (st, [cfgp, _P, _P, _P, _P]),
        "moe_dispatch": (st, [cfgp, _P, _P, _P, _P, _P, _P, _P, _P, _P, sz, _P]),
        "moe_dispatch_noalloc": (st, [cfgp, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
        "moe_ffn_up": (st, [cfgp, _P, _P, _P, _P, _P, _P, sz, _P]),
        "moe_ffn_up_gather": (st, [cfgp, _P, _P, _P, _P, _P, _P, _P, sz, _P]),
        "moe_ffn_down": (st, [cfgp, _P, _P, _P, _P, _P, _P, sz, _P]),
        "moe_ffn_down_combine": (st, [cfgp, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, sz, _P]),
        "moe_expert_ffn": (st, [cfgp, _P, _P, _P, _P, _P, _P, _P, _P, _P, sz, _P]),
        "moe_combine": (st, [cfgp, _P, _P, _P, _P, _P]),
        "moe_aux_stats": (st, [cfgp, _P, _P, ctypes.c_float, _P, _P, _P, _P]),
        "moe_forward": (st, [cfgp, ctypes.POINTER(Tensors), ctypes.c_float, _P, sz, _P]),
        "moe_get_device_status": (st, [_P, ctypes.POINTER(ctypes.c_int32)]),
        "moe_selftest_wait_timeout": (st, [_P, sz, i64, _P]),
        "moe_selftest_grid_barrier_timeout": (st, [_P, sz, i64, _P]),
        "moe_launch_count": (i64, []),
        "moe_status_string": (ctypes.c_char_p, [st]),
        "moe_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _status_name(code):
    try:
        return load().moe_status_string(code).decode()
    except Exception:  # noqa: BLE001 - only for the message
        return str(code)


def _check(code):
    if code != MOE_OK:
        raise MoeError(code, load().moe_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmoe takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libmoe takes contiguous tensors")
    return _P(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return _P(s.cuda_stream)


def config(T, d, d_ff, E, k, capacity_factor, renormalize=True, act="gelu_tanh", dtype="bf16",
           write_logits=False, reroute=False, fuse_dispatch=False, fuse_combine=False) -> Config:
    return Config(T=T, d=d, d_ff=d_ff, E=E, k=k, capacity_factor=float(capacity_factor),
                  renormalize=int(bool(renormalize)),
                  act=MOE_ACT_RELU if act == "relu" else MOE_ACT_GELU_TANH,
                  dtype=MOE_DT_BF16 if dtype == "bf16" else MOE_DT_F32,
                  write_logits=int(bool(write_logits)), reroute=int(bool(reroute)),
                  fuse_dispatch=int(bool(fuse_dispatch)), fuse_combine=int(bool(fuse_combine)))


def config_from_workload(wl, write_logits=False, reroute=False, fuse_dispatch=False,
                         fuse_combine=False) -> Config:
    return config(wl.T, wl.d, wl.d_ff, wl.E, wl.k, wl.capacity_factor, wl.renormalize, wl.act,
                  wl.dtype, write_logits, reroute, fuse_dispatch, fuse_combine)


def capacity(cfg: Config) -> int:
    c = load().moe_capacity(ctypes.byref(cfg))
    if c < 0:
        _check(MOE_ERR_INVALID_ARG)
    return int(c)


def max_rows(cfg: Config) -> int:
    r = load().moe_max_rows(ctypes.byref(cfg))
    if r < 0:
        _check(MOE_ERR_INVALID_ARG)
    return int(r)


def workspace_size(cfg: Config) -> int:
    n = ctypes.c_size_t(0)
    _check(load().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return int(n.value)


def act_dtype(cfg: Config):
    return torch.bfloat16 if cfg.dtype == MOE_DT_BF16 else torch.float32


def workspace(cfg: Config, device="cuda", stream=None) -> torch.Tensor:
    """Allocate (through torch) and clear a workspace for cfg."""
    ws = torch.empty(workspace_size(cfg), dtype=torch.uint8, device=device)
    _check(load().moe_workspace_init(_ptr(ws), ws.numel(), _stream(stream)))
    return ws


def allocate(cfg: Config, device="cuda", health: bool = False) -> dict:
    """Allocate every output and intermediate tensor of one forward pass
    (``health``: also the 4 routing-health indicators, which forward() then
    computes; with ``cfg.fuse_dispatch`` there is no dispatch buffer xd)."""
    dt = act_dtype(cfg)
    T, d, d_ff, E, k = cfg.T, cfg.d, cfg.d_ff, cfg.E, cfg.k
    R = max(max_rows(cfg), 1)
    z = dict(device=device)
    return dict(
        logits=torch.empty((T, E), dtype=torch.float32, **z) if cfg.write_logits else None,
        topk_ids=torch.empty((T, k), dtype=torch.int32, **z),
        topk_w=torch.empty((T, k), dtype=torch.float32, **z),
        psum=torch.empty(E, dtype=torch.float32, **z),
        counts=torch.empty(E, dtype=torch.int32, **z),
        kept=torch.empty(E, dtype=torch.int32, **z),
        offsets=torch.empty(E + 1, dtype=torch.int32, **z),
        slot_row=torch.empty((T, k), dtype=torch.int32, **z),
        row_token=torch.empty(R, dtype=torch.int32, **z),
        xd=None if cfg.fuse_dispatch else torch.empty((R, d), dtype=dt, **z),
        H=torch.empty((R, d_ff), dtype=dt, **z),
        yd=torch.empty((R, d), dtype=dt, **z),
        y=torch.empty((T, d), dtype=dt, **z),
        f=torch.empty(E, dtype=torch.float32, **z),
        pbar=torch.empty(E, dtype=torch.float32, **z),
        l_aux=torch.empty(1, dtype=torch.float32, **z),
        health=torch.empty(4, dtype=torch.float32, **z) if health else None,
    )


def route(cfg, x, Wr, br, out, ws, stream=None, sel_bias=None):
    """moe_route, or moe_route_sel when ``sel_bias`` (fp32 [E]) is given."""
    if sel_bias is None:
        _check(load().moe_route(ctypes.byref(cfg), _ptr(x), _ptr(Wr), _ptr(br),
                                _ptr(out.get("logits")), _ptr(out["topk_ids"]),
                                _ptr(out["topk_w"]), _ptr(out["psum"]), _ptr(ws), ws.numel(),
                                _stream(stream)))
    else:
        _check(load().moe_route_sel(ctypes.byref(cfg), _ptr(x), _ptr(Wr), _ptr(br),
                                    _ptr(sel_bias), _ptr(out.get("logits")),
                                    _ptr(out["topk_ids"]), _ptr(out["topk_w"]),
                                    _ptr(out["psum"]), _ptr(ws), ws.numel(), _stream(stream)))


def routing_health(cfg, counts, kept, health, stream=None):
    """moe_routing_health: health[4] from counts and kept."""
    _check(load().moe_routing_health(ctypes.byref(cfg), _ptr(counts), _ptr(kept), _ptr(health),
                                     _stream(stream)))


def dispatch(cfg, x, topk_ids, out, ws, stream=None):
    _check(load().moe_dispatch(ctypes.byref(cfg), _ptr(x), _ptr(topk_ids), _ptr(out["counts"]),
                               _ptr(out["kept"]), _ptr(out["offsets"]), _ptr(out["slot_row"]),
                               _ptr(out["row_token"]), _ptr(out.get("xd")), _ptr(ws), ws.numel(),
                               _stream(stream)))


def dispatch_noalloc(cfg, x, topk_ids, out, status=None, stream=None):
    """moe_dispatch without a workspace (scratch in a fixed library array)."""
    _check(load().moe_dispatch_noalloc(ctypes.byref(cfg), _ptr(x), _ptr(topk_ids),
                                       _ptr(out["counts"]), _ptr(out["kept"]),
                                       _ptr(out["offsets"]), _ptr(out["slot_row"]),
                                       _ptr(out["row_token"]), _ptr(out.get("xd")), _ptr(status),
                                       _stream(stream)))


def ffn_up(cfg, xd, offsets, W1, b1, H, ws, stream=None):
    _check(load().moe_ffn_up(ctypes.byref(cfg), _ptr(xd), _ptr(offsets), _ptr(W1), _ptr(b1),
                             _ptr(H), _ptr(ws), ws.numel(), _stream(stream)))


def ffn_up_gather(cfg, x, row_token, offsets, W1, b1, H, ws, stream=None):
    """moe_ffn_up_gather: the first GEMM on the rows x[row_token[row]]."""
    _check(load().moe_ffn_up_gather(ctypes.byref(cfg), _ptr(x), _ptr(row_token), _ptr(offsets),
                                    _ptr(W1), _ptr(b1), _ptr(H), _ptr(ws), ws.numel(),
                                    _stream(stream)))


def ffn_down(cfg, H, offsets, W2, b2, yd, ws, stream=None):
    _check(load().moe_ffn_down(ctypes.byref(cfg), _ptr(H), _ptr(offsets), _ptr(W2), _ptr(b2),
                               _ptr(yd), _ptr(ws), ws.numel(), _stream(stream)))


def ffn_down_combine(cfg, H, offsets, row_token, slot_row, topk_w, W2, b2, yd, y, ws,
                     stream=None):
    """moe_ffn_down_combine: the second GEMM with the combine in its epilogue."""
    _check(load().moe_ffn_down_combine(ctypes.byref(cfg), _ptr(H), _ptr(offsets), _ptr(row_token),
                                       _ptr(slot_row), _ptr(topk_w), _ptr(W2), _ptr(b2),
                                       _ptr(yd), _ptr(y), _ptr(ws), ws.numel(), _stream(stream)))


def expert_ffn(cfg, xd, offsets, W1, b1, W2, b2, H, yd, ws, stream=None):
    _check(load().moe_expert_ffn(ctypes.byref(cfg), _ptr(xd), _ptr(offsets), _ptr(W1), _ptr(b1),
                                 _ptr(W2), _ptr(b2), _ptr(H), _ptr(yd), _ptr(ws), ws.numel(),
                                 _stream(stream)))


def combine(cfg, yd, slot_row, topk_w, y, stream=None):
    _check(load().moe_combine(ctypes.byref(cfg), _ptr(yd), _ptr(slot_row), _ptr(topk_w), _ptr(y),
                              _stream(stream)))


def aux_stats(cfg, counts, psum, alpha, f, pbar, l_aux, stream=None):
    _check(load().moe_aux_stats(ctypes.byref(cfg), _ptr(counts), _ptr(psum), float(alpha),
                                _ptr(f), _ptr(pbar), _ptr(l_aux), _stream(stream)))


def tensors_struct(inputs: dict, out: dict) -> Tensors:
    t = Tensors()
    for name in _TENSOR_FIELDS:
        src = inputs.get(name) if name in inputs else out.get(name)
        setattr(t, name, None if src is None else _ptr(src).value)
    return t


def forward(cfg, inputs: dict, out: dict, ws, alpha=0.01, stream=None):
    """The whole layer in one library call (route, dispatch, FFN, combine, aux)."""
    t = tensors_struct(inputs, out)
    _check(load().moe_forward(ctypes.byref(cfg), ctypes.byref(t), float(alpha), _ptr(ws),
                              ws.numel(), _stream(stream)))


def forward_stages(cfg, inputs: dict, out: dict, ws, alpha=0.01, stream=None, events=None):
    """The same launches as forward(), one stage call at a time.

    ``events``: optional list of 7 CUDA events recorded on the stream before
    route, dispatch, ffn_up, ffn_down, combine, aux and after aux.
    """
    s = stream if stream is not None else torch.cuda.current_stream()

    def mark(i):
        if events is not None:
            events[i].record(s)

    mark(0)
    route(cfg, inputs["x"], inputs["Wr"], inputs["br"], out, ws, s,
          sel_bias=inputs.get("sel_bias"))
    mark(1)
    dispatch(cfg, inputs["x"], out["topk_ids"], out, ws, s)
    mark(2)
    if cfg.fuse_dispatch:
        ffn_up_gather(cfg, inputs["x"], out["row_token"], out["offsets"], inputs["W1"],
                      inputs["b1"], out["H"], ws, s)
    else:
        ffn_up(cfg, out["xd"], out["offsets"], inputs["W1"], inputs["b1"], out["H"], ws, s)
    mark(3)
    if cfg.fuse_combine:
        ffn_down_combine(cfg, out["H"], out["offsets"], out["row_token"], out["slot_row"],
                         out["topk_w"], inputs["W2"], inputs["b2"], out["yd"], out["y"], ws, s)
    else:
        ffn_down(cfg, out["H"], out["offsets"], inputs["W2"], inputs["b2"], out["yd"], ws, s)
    mark(4)
    if not cfg.fuse_combine:
        combine(cfg, out["yd"], out["slot_row"], out["topk_w"], out["y"], s)
    mark(5)
    aux_stats(cfg, out["counts"], out["psum"], alpha, out["f"], out["pbar"], out["l_aux"], s)
    if out.get("health") is not None:
        routing_health(cfg, out["counts"], out["kept"], out["health"], s)
    mark(6)


def selftest_wait_timeout(ws, limit_ns: int, stream=None):
    """moe_selftest_wait_timeout: a bounded wait that must give up and record
    MOE_ERR_TIMEOUT in the workspace status word."""
    _check(load().moe_selftest_wait_timeout(_ptr(ws), ws.numel(), int(limit_ns), _stream(stream)))


def selftest_grid_barrier_timeout(ws, limit_ns: int, stream=None):
    """moe_selftest_grid_barrier_timeout: the one-pass dispatch's grid barrier
    waiting for a block that never arrives must give up and record
    MOE_ERR_TIMEOUT in the workspace status word."""
    _check(load().moe_selftest_grid_barrier_timeout(_ptr(ws), ws.numel(), int(limit_ns),
                                                    _stream(stream)))


def workspace_init(ws, stream=None):
    """Clear a workspace's header (status word, counters, accumulators)."""
    _check(load().moe_workspace_init(_ptr(ws), ws.numel(), _stream(stream)))


def device_status(ws) -> int:
    """Status word of a workspace (blocking read; synchronise the stream first)."""
    v = ctypes.c_int32(0)
    _check(load().moe_get_device_status(_ptr(ws), ctypes.byref(v)))
    return int(v.value)


def launch_count() -> int:
    return int(load().moe_launch_count())


@dataclass
class Layer:
    """A configured layer with its workspace and output buffers on one device."""
    cfg: Config
    ws: torch.Tensor
    out: dict

    @classmethod
    def create(cls, cfg: Config, device="cuda"):
        return cls(cfg, workspace(cfg, device), allocate(cfg, device))

    def __call__(self, inputs: dict, alpha=0.01, stream=None):
        forward(self.cfg, inputs, self.out, self.ws, alpha, stream)
        return self.out
