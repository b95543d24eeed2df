"""The benchmark's multi-rank logic on CPU: two gloo ranks (world size 2,
127.0.0.1) run independent replicas, and the job's time is the slowest
rank's.  No GPU: only the host-side aggregation is exercised."""

import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # Each replica measured its own time; the job reports the slowest.
        local_ms = 10.0 + 5.0 * rank
        max_ms = bench.max_over_ranks(local_ms, dist)
        dist.barrier()
        value = bench.job_tokens_per_s(world, 4096, 3, max_ms)
        q.put((rank, max_ms, value, bench.replica_seed(7, rank)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]
    want = 2 * 4096 * 3 / 15e-3
    assert all(abs(r[2] - want) <= 1e-9 * want for r in res)
    # every replica routes its own batch
    assert res[0][3] != res[1][3]


def test_single_process_aggregation_is_the_identity():
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.job_tokens_per_s(1, 4096, 20, 3.2) == pytest.approx(4096 * 20 / 3.2e-3)


def test_reference_arm_runs_on_rank_zero_only():
    # Under torchrun the reference arm prints from rank 0; the other ranks
    # exit 0 without work (they never touch the workload).
    assert bench.run_reference(None, None, rank=1, world=2) == 0
