"""The N > 1 host logic of bench.py, on CPU with world-size-2 gloo process
groups: every rank runs its own replica (weak scaling, no collective on the
data path); the timed milliseconds are the maximum over ranks, the rate is the
units all ranks processed over that time, and only rank 0 reports."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sock:
        sock.bind(("127.0.0.1", 0))
        return sock.getsockname()[1]


def _rank_main(rank, world, port, local_ms, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(local_ms[rank], world, torch.device("cpu"))
        rate = bench.whole_job_rate(1000.0, 10, world, ms)
        results[rank] = (ms, rate)
    finally:
        dist.destroy_process_group()


def _run(world, local_ms):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as manager:
        results = manager.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, local_ms, results))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0, f"rank exited with {p.exitcode}"
        return dict(results)


def test_max_over_ranks_and_whole_job_rate_gloo_world_2():
    out = _run(2, [12.5, 40.0])
    assert set(out) == {0, 1}
    for rank in (0, 1):
        ms, rate = out[rank]
        assert ms == 40.0                                   # the slowest rank sets the time
        assert rate == pytest.approx(1000.0 * 10 * 2 / 0.040)   # units of both ranks


def test_single_rank_needs_no_process_group():
    import torch

    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.25, 1, torch.device("cpu")) == 7.25
    assert bench.whole_job_rate(16.0, 4, 1, 8.0) == pytest.approx(16.0 * 4 / 0.008)


def test_reference_arm_only_rank_0_works(capsys):
    """Under torchrun the reference arm runs on rank 0 alone; other ranks
    return at once without work or output."""
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        workload, steps, warmup, reference_rows = "tiny", 1, 0, 4
    assert bench.run_reference(Args(), rank=1, world=2) is None
    assert capsys.readouterr().out == ""
