"""Multi-rank host logic of the benchmark, on the CPU with gloo.

The op has no exchange step, so N GPUs run N independent replicas: every
rank times its own steps, the job's time is the slowest rank's, and the
reported value counts the tokens of all ranks (weak scaling).  Two gloo ranks
drive the same helpers that bench.py uses under torchrun (process group from
the environment, barrier, max over ranks, whole-job throughput); the
reference arm runs on rank 0 alone and the other ranks exit without work.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, seconds, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    w, r, local = bench.setup_dist(backend="gloo")
    bench.barrier(w, cuda=False)
    t = bench.max_over_ranks(seconds[rank], w, device="cpu")
    value = bench.job_throughput(256, w, 10, t)
    out_q.put((r, w, local, t, value))
    bench.barrier(w, cuda=False)
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_all_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    seconds = [1.5, 2.0]  # rank 1 is the slow one
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, seconds, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=180) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, (r, w, local, t, value) in enumerate(got):
        assert (r, w, local) == (rank, 2, rank)
        assert t == 2.0                                    # the max over ranks
        assert value == pytest.approx(256 * 2 * 10 / 2.0)  # tokens of both replicas


def test_job_throughput_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_throughput(256, 1, 10, 2.0)
    assert bench.job_throughput(256, 4, 10, 2.0) == pytest.approx(4 * one)
    assert bench.max_over_ranks(3.25, 1) == 3.25  # one rank: no process group


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""
