"""The multi-rank host logic of bench.py on CPU: world_size 2 over gloo (the
data path has no collective; ranks meet only to take the slowest rank's time),
and the reference arm's rank gating."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    # per-rank timings that differ: every rank must see the maximum
    vals = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)], world)
    q.put((rank, vals, bench.job_throughput(10.0, world, vals[0])))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict()
    for _ in range(2):
        rank, vals, rate = q.get(timeout=120)
        out[rank] = (vals, rate)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        vals, rate = out[rank]
        assert vals == [2.0, 5.0, 0.5]
        assert rate == pytest.approx(2 * 10.0 / 2e-3)


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup = 1, 1

    bench.run_reference(A)  # rank 1: returns at once, prints nothing
    assert capsys.readouterr().out == ""
