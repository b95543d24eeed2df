"""The C-ABI library loads and exports every declared entry point; its
host-only functions (capacity, buffer sizes, argument checks) behave as the
header states.  CPU only: nothing here launches a kernel."""

import ctypes
import math
import os
import re
from fractions import Fraction

import pytest

import oracle
from routing_dispatch_expert_06_b300 import build as moe_build
from routing_dispatch_expert_06_b300 import moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward",
                     "moe_aux_stats"]:
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def cfg_for(T, d, d_ff, E, k, c, **kw):
    return moe.config(T, d, d_ff, E, k, c, **kw)


@pytest.mark.parametrize("T,k,E,c", [(8, 1, 2, 1.0), (8, 1, 2, 1.5), (1024, 1, 8, 1.25),
                                     (1024, 1, 8, 2.0), (512, 2, 8, 1.0), (4096, 2, 8, 1.25),
                                     (16384, 1, 8, 1.0), (8192, 6, 64, 1.0),
                                     (32768, 8, 256, 1.25), (10, 1, 1, 1.1), (7, 3, 5, 0.3)])
def test_capacity_matches_definition(lib, T, k, E, c):
    cfg = cfg_for(T, 64, 64, E, k, c)
    C = moe.capacity(cfg)
    assert C == math.ceil(Fraction(c) * T * k / E)
    assert C == oracle.capacity(T, k, E, c)
    assert moe.max_rows(cfg) == min(T * k, E * C)


def test_workspace_size_positive_and_aligned(lib):
    for T, E in [(1, 1), (512, 8), (32768, 256), (100000, 1024)]:
        n = moe.workspace_size(cfg_for(T, 64, 64, E, 1, 1.0))
        assert n > 0 and n % 256 == 0


@pytest.mark.parametrize("bad", [
    dict(T=0), dict(E=0), dict(E=1025), dict(k=0), dict(k=17), dict(E=4, k=5), dict(d=12),
    dict(d_ff=20), dict(capacity_factor=0.0), dict(capacity_factor=-1.0),
    dict(T=1 << 28, k=8)])
def test_invalid_config_rejected(lib, bad):
    base = dict(T=64, d=64, d_ff=64, E=8, k=2, capacity_factor=1.0)
    base.update(bad)
    cfg = moe.config(**base)
    n = ctypes.c_size_t(0)
    assert lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_capacity(ctypes.byref(cfg)) == -1
    assert lib.moe_last_error().decode() != ""


def test_unsupported_dtype_and_act(lib):
    cfg = cfg_for(64, 64, 64, 8, 2, 1.0)
    cfg.dtype = 7
    n = ctypes.c_size_t(0)
    assert lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == moe.MOE_ERR_UNSUPPORTED
    cfg = cfg_for(64, 64, 64, 8, 2, 1.0)
    cfg.act = 9
    assert lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == moe.MOE_ERR_UNSUPPORTED


def test_null_tensors_rejected_before_any_launch(lib):
    cfg = cfg_for(64, 64, 64, 8, 2, 1.0)
    P = ctypes.c_void_p
    ws = P(256)  # never dereferenced: the NULL check comes first
    assert lib.moe_route(ctypes.byref(cfg), None, None, None, None, None, None, None, ws, 1 << 20,
                         None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch(ctypes.byref(cfg), None, None, None, None, None, None, None, None, ws,
                            1 << 20, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(ctypes.byref(cfg), None, None, None, None, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert lib.moe_aux_stats(ctypes.byref(cfg), None, None, 1.0, None, None, None, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert lib.moe_forward(ctypes.byref(cfg), None, 1.0, ws, 1 << 20, None) == \
        moe.MOE_ERR_INVALID_ARG


def test_small_workspace_rejected(lib):
    cfg = cfg_for(4096, 64, 64, 8, 2, 1.0)
    P = ctypes.c_void_p
    need = moe.workspace_size(cfg)
    fake = P(1 << 12)  # aligned, never dereferenced
    r = lib.moe_route(ctypes.byref(cfg), P(16), P(16), P(16), None, P(16), P(16), P(16), fake,
                      need - 256, None)
    assert r == moe.MOE_ERR_WORKSPACE


def test_status_strings(lib):
    for code, name in [(0, "MOE_OK"), (1, "MOE_ERR_INVALID_ARG"), (5, "MOE_ERR_TIMEOUT")]:
        assert lib.moe_status_string(code).decode() == name


def test_reroute_flag_checked_and_sized(lib):
    # reroute must be 0 or 1; with it the workspace grows by the candidate,
    # offer and position arrays (4 × T·k int32) and two [E] arrays.
    base = cfg_for(4096, 1024, 4096, 8, 2, 1.25)
    rr = cfg_for(4096, 1024, 4096, 8, 2, 1.25, reroute=True)
    n0, n1 = moe.workspace_size(base), moe.workspace_size(rr)
    assert n1 - n0 >= 4 * 4096 * 2 * 4 + 2 * 8 * 4
    bad = cfg_for(64, 64, 64, 8, 2, 1.0)
    bad.reroute = 2
    n = ctypes.c_size_t(0)
    assert lib.moe_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == moe.MOE_ERR_INVALID_ARG


def test_workspace_header_holds_the_column_sum_accumulators(lib):
    # moe_workspace_init clears the header; the smallest valid workspace is at
    # least that large (status word, counters, 32 × 1024 uint64 accumulators).
    assert moe.workspace_size(cfg_for(1, 8, 8, 1, 1, 1.0)) >= 16384 + 32 * 1024 * 8


def test_new_entry_points_reject_null_arguments(lib):
    cfg = cfg_for(64, 64, 64, 8, 2, 1.0)
    assert lib.moe_routing_health(ctypes.byref(cfg), None, None, None, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert lib.moe_route_sel(ctypes.byref(cfg), None, None, None, None, None, None, None, None,
                             None, 0, None) == moe.MOE_ERR_INVALID_ARG


def test_selftest_rejects_bad_arguments(lib):
    assert lib.moe_selftest_wait_timeout(None, 0, 10**7, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_grid_barrier_timeout(None, 0, 10**7, None) == \
        moe.MOE_ERR_INVALID_ARG


def test_fuse_dispatch_flag_and_gather_scope(lib):
    # fuse_dispatch must be 0 or 1.  The gathering first GEMM exists for bf16
    # layers on the regular tensor-core GEMM only: fp32 layers and layers with
    # at most 64 rows per expert get MOE_ERR_UNSUPPORTED before any launch
    # (the placeholder pointers below are never dereferenced).
    bad = cfg_for(64, 64, 64, 8, 2, 1.0)
    bad.fuse_dispatch = 2
    n = ctypes.c_size_t(0)
    assert lib.moe_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == moe.MOE_ERR_INVALID_ARG
    ok = cfg_for(4096, 1024, 4096, 8, 2, 1.25, fuse_dispatch=True)
    assert lib.moe_ffn_up_gather(ctypes.byref(ok), None, None, None, None, None, None, None, 0,
                                 None) == moe.MOE_ERR_INVALID_ARG
    p = ctypes.c_void_p(1 << 20)
    f32 = cfg_for(4096, 1024, 4096, 8, 2, 1.25, dtype="f32", fuse_dispatch=True)
    dec = cfg_for(8, 2048, 1408, 64, 6, 1.0, fuse_dispatch=True)  # min(C, T·k) = 1
    for cfg in (f32, dec):
        assert lib.moe_ffn_up_gather(ctypes.byref(cfg), p, p, p, p, p, p, p, 1 << 30,
                                     None) == moe.MOE_ERR_UNSUPPORTED


def test_fuse_dispatch_host_checks(lib):
    # moe_dispatch takes a NULL xd only with fuse_dispatch: without it the call
    # is refused as a NULL tensor; with it the call gets past the tensor checks
    # and stops at the (too small) workspace, before any launch.  moe_forward
    # refuses fuse_dispatch on an fp32 layer before any launch.
    p = ctypes.c_void_p(1 << 20)
    cfg = cfg_for(4096, 1024, 4096, 8, 2, 1.25)
    args = [p] * 7 + [None, p, 16]  # x, ids, counts, kept, offsets, slot_row, row_token, xd, ws
    assert lib.moe_dispatch(ctypes.byref(cfg), *args, None) == moe.MOE_ERR_INVALID_ARG
    fused = cfg_for(4096, 1024, 4096, 8, 2, 1.25, fuse_dispatch=True)
    assert lib.moe_dispatch(ctypes.byref(fused), *args, None) == moe.MOE_ERR_WORKSPACE
    f32 = cfg_for(512, 128, 512, 8, 2, 1.0, dtype="f32", fuse_dispatch=True)
    t = moe.Tensors()
    for name in ("f", "pbar", "l_aux"):
        setattr(t, name, 1 << 20)
    assert lib.moe_forward(ctypes.byref(f32), ctypes.byref(t), ctypes.c_float(1.0), p, 1 << 30,
                           None) == moe.MOE_ERR_UNSUPPORTED


def test_fuse_combine_flag_scope_and_counters(lib):
    # fuse_combine must be 0 or 1; it adds 2 int32 counters per token and
    # 256-wide column tile of d to the workspace; moe_ffn_down_combine refuses
    # NULL tensors, a config without the flag (no counters) and the layers the
    # tensor-core GEMM does not run (fp32, at most 64 rows per expert), all
    # before any launch (the placeholder pointers are never dereferenced).
    bad = cfg_for(64, 64, 64, 8, 2, 1.0)
    bad.fuse_combine = 2
    n = ctypes.c_size_t(0)
    assert lib.moe_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == moe.MOE_ERR_INVALID_ARG
    plain = cfg_for(32768, 7168, 2048, 256, 8, 1.25)
    fused = cfg_for(32768, 7168, 2048, 256, 8, 1.25, fuse_combine=True)
    assert moe.workspace_size(fused) - moe.workspace_size(plain) >= 32768 * 2 * 28 * 4
    p = ctypes.c_void_p(1 << 20)
    args = [p] * 9 + [p, 1 << 30, None]
    assert lib.moe_ffn_down_combine(ctypes.byref(fused), *([None] * 9), p, 1 << 30,
                                    None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_ffn_down_combine(ctypes.byref(plain), *args) == moe.MOE_ERR_INVALID_ARG
    f32 = cfg_for(4096, 1024, 4096, 8, 2, 1.25, dtype="f32", fuse_combine=True)
    dec = cfg_for(8, 2048, 1408, 64, 6, 1.0, fuse_combine=True)
    for cfg in (f32, dec):
        assert lib.moe_ffn_down_combine(ctypes.byref(cfg), *args) == moe.MOE_ERR_UNSUPPORTED
