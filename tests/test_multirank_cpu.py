"""The benchmark's multi-process host logic on CPU: two ranks over the gloo backend.

Each rank runs its own replica of the workload (no exchange on the data path), so the
only cross-rank steps are the barriers around the timed region and the reduction of the
time to the slowest rank.  Checked here: every rank gets the slowest rank's time, the
whole-job value counts all ranks' work over that time, and in the reference arm only
rank 0 does any work or prints.
"""

import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        t = bench.max_over_ranks(local_ms[rank], world, "cpu")
        value = bench.job_tflops(1e12, 10, world, t)
        out[rank] = (t, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_all_work():
    world, local_ms = 2, [40.0, 50.0]
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, local_ms, out), nprocs=world,
                           join=True, start_method="spawn")
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in range(world):
        t, value = res[rank]
        assert t == 50.0                    # the slowest rank's time, on every rank
        # 10 steps of 1 TFLOP on each of 2 ranks in 50 ms
        assert value == pytest.approx(2 * 10 * 1.0 / 0.050)


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.job_tflops(2e12, 5, 1, 100.0) == pytest.approx(100.0)


def test_reference_arm_runs_on_rank_0_only(monkeypatch):
    """Under torchrun the reference arm's other ranks exit at once, without work or output."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2",
                                      "--steps", "1", "--warmup", "3"])
    called = []
    monkeypatch.setattr(bench, "run_reference", lambda *a: called.append(a))
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main()
    assert called == []
    assert buf.getvalue() == ""
