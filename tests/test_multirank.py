"""Multi-rank logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

The path shards by rows with no data exchange; the only cross-rank steps are
the barrier around the timed region and the max-over-ranks of the times.
Each rank here reports a different time; both must see the largest, and the
whole-job rate must count every rank's units over that time.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            init_method=f"tcp://127.0.0.1:{port}")
    try:
        bench.barrier(world)
        local_ms = 100.0 + 25.0 * rank  # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
        rate = bench.job_rate(1000, world, ms, steps=10)
        bench.barrier(world)
        out.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_every_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(2):
        rank, ms, rate = out.get(timeout=120)
        got[rank] = (ms, rate)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see rank 1's 125 ms; 2 ranks x 1000 units per step, 10 steps
    for rank in (0, 1):
        ms, rate = got[rank]
        assert ms == 125.0
        assert rate == pytest.approx(2 * 1000 / (125.0 / 10 / 1e3))


def test_one_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    bench.barrier(1)
    assert bench.max_over_ranks(42.0, 1, torch.device("cpu")) == 42.0
    assert bench.job_rate(512, 1, 2.0, steps=4) == pytest.approx(512 / 0.0005)
