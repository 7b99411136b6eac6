"""The multi-rank bookkeeping of bench.py on CPU: two gloo ranks (127.0.0.1) reduce their step times to the
slowest rank's, and the whole-job rate counts every rank's rows in that time (weak scaling, replicas)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                                         world_size=world)
    try:
        ms = bench.max_over_ranks(1.0 + rank, world, "cpu")   # rank 1 is the slower one
        q.put((rank, ms, bench.job_rate(8192, ms, world)))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_every_rank():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, rate in got:
        assert ms == 2.0
        assert rate == pytest.approx(2 * 8192 / 2e-3)


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_rate(8192, 0.5, 1) == pytest.approx(8192 / 0.5e-3)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    """Under torchrun the reference arm (the oracle on the host cores) runs on rank 0; other ranks exit
    without work."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(None, None) is None
