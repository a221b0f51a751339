"""Host logic of bench.py's N > 1 path, on CPU with gloo (world size 2).

The path is replicas only: every rank runs the same step on its own GPU and
no data-path collective exists; the ranks meet only to take the slowest
rank's time, and `value` is the work of all ranks over that time.  The
reference arm runs on rank 0 alone.
"""
import os
import socket
import types

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(dist, times[rank], "cpu")
        q.put((rank, ms, bench.whole_job_tflops(2.0e12, world, 4, ms)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_time_and_whole_job_value_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [12.5, 20.0]
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in got:
        assert ms == 20.0  # every rank sees the slowest rank's time
        # 2 ranks x 4 steps x 2 TFLOP in 20 ms
        assert value == pytest.approx(2.0e12 * 2 * 4 / 0.020 / 1e12)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(None, 7.25, "cpu") == 7.25
    assert bench.whole_job_tflops(1.0e12, 1, 10, 1000.0) == pytest.approx(10.0)


def test_reference_arm_runs_on_rank_zero_only():
    args = types.SimpleNamespace(warmup=1, steps=1)
    # a rank other than 0 returns at once, touching neither the oracle nor the workload
    assert bench.run_reference(args, None, 2, 1) == 0
