"""bench.py's multi-rank host logic on CPU: two gloo ranks, the slowest rank's time and the
whole-job throughput, and the reference arm staying on rank 0."""
import os
import socket
import sys

import torch
import torch.multiprocessing as mp

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = (3.0, 5.0)[rank]  # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, "cpu")
        q.put((rank, slowest, bench.job_throughput(100.0, world, slowest)))
        torch.distributed.barrier()
    finally:
        torch.distributed.destroy_process_group()


def test_two_ranks_report_the_slowest_time_and_all_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == 5.0
        assert value == 100.0 * 2 / 5e-3


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(7.5, "cpu") == 7.5
    assert bench.job_throughput(10.0, 1, 2.0) == 5000.0


def test_reference_arm_runs_on_rank_0_only(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference"])
    assert bench.run_reference(bench.parse(), 1) is None
