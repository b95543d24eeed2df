"""Every stage call of the C ABI opens an NVTX range named after it (a
profiler's timeline then shows the stages of a forward pass by name).  CPU
only: a small NVTX tool (tests/nvtx_injection.c) records the ranges while a
child process makes calls that fail their argument checks, so no kernel runs."""

import os
import shutil
import subprocess
import sys

import pytest

from routing_dispatch_expert_06_b300 import build as moe_build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CALLS = ["moe_route", "moe_route_sel", "moe_dispatch", "moe_dispatch_noalloc", "moe_ffn_up",
         "moe_ffn_up_gather", "moe_ffn_down", "moe_combine", "moe_aux_stats",
         "moe_routing_health", "moe_forward"]

CHILD = r"""
import ctypes, sys
from routing_dispatch_expert_06_b300 import moe
lib = moe.load()
cfg = moe.config(64, 64, 64, 8, 2, 1.0)

def null_args(fn):
    args = [ctypes.byref(cfg)]
    for t in fn.argtypes[1:]:
        if t in (ctypes.c_size_t, ctypes.c_int64, ctypes.c_int32):
            args.append(0)
        elif t is ctypes.c_float:
            args.append(0.0)
        else:
            args.append(None)
    return args

for name in sys.argv[1:]:
    fn = getattr(lib, name)
    assert fn(*null_args(fn)) == moe.MOE_ERR_INVALID_ARG, name
"""


@pytest.fixture(scope="module")
def injection(tmp_path_factory):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    moe_build.build()
    out = tmp_path_factory.mktemp("nvtx") / "libnvtx_injection.so"
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    subprocess.run([gcc, "-shared", "-fPIC", "-O1", "-I", cuda_inc,
                    os.path.join(HERE, "nvtx_injection.c"), "-o", str(out)], check=True)
    return str(out)


def test_each_stage_call_opens_a_named_range(injection, tmp_path):
    log = tmp_path / "ranges.txt"
    env = dict(os.environ, NVTX_INJECTION64_PATH=injection, MOE_NVTX_LOG=str(log),
               PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    subprocess.run([sys.executable, "-c", CHILD, *CALLS], check=True, env=env, cwd=ROOT,
                   timeout=120)
    lines = log.read_text().split("\n")[:-1]
    pushes = [ln[5:] for ln in lines if ln.startswith("push ")]
    # moe_route_sel runs the router under the name of the stage, moe_route
    assert pushes == [c if c != "moe_route_sel" else "moe_route" for c in CALLS]
    assert lines.count("pop") == len(pushes)
    # ranges close in order: every push is followed by its pop
    assert lines == [x for c in pushes for x in (f"push {c}", "pop")]
