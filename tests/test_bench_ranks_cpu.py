"""Multi-rank bookkeeping of bench.py on CPU: two gloo ranks stand in for two
GPUs running replicas of the step.  The job's time is the slowest rank's and
the job's throughput counts every rank's work; the reference arm prints only
on rank 0."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, ms_by_rank, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import sys
        sys.path.insert(0, ROOT)  # a spawned process does not run conftest
        import bench
        t = bench.max_over_ranks(ms_by_rank[rank], dist, torch.device("cpu"))
        out.put((rank, t, bench.job_tflops(bench.STEP_FLOP, world, t)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_all_work():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    ms = [1.25, 1.5]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, ms, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import bench
    want_value = 2 * bench.STEP_FLOP / 1.5e-3 / 1e12
    for rank, t, v in got:
        assert t == 1.5, rank
        assert v == pytest.approx(want_value, rel=1e-12)


def test_single_rank_keeps_its_own_time():
    import bench
    assert bench.max_over_ranks(2.5, None, torch.device("cpu")) == 2.5
    assert bench.job_tflops(bench.STEP_FLOP, 1, 1.0) == pytest.approx(bench.STEP_FLOP / 1e-3 / 1e12)


def test_reference_arm_prints_only_on_rank_zero(capsys, monkeypatch):
    import bench

    class Args:
        steps, warmup = 1, 0

    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(Args())
    assert capsys.readouterr().out == ""
