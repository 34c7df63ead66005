"""Multi-GPU is replicas only: each rank decodes its own stream and the job's
throughput is (ranks x steps) / (slowest rank's time).  This checks the
benchmark's aggregation with two gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.slowest_rank_ms(times[rank], world)
        out[rank] = (ms, bench.replica_tok_s(world, 128, ms))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, times = 2, [2.5, 3.0]  # ms per 128 steps on each rank
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms, tok_s = res[r]
        assert ms == 3.0                                   # every rank sees the max
        assert tok_s == pytest.approx(2 * 128 / 3.0e-3)   # total over both replicas


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    assert bench.slowest_rank_ms(1.25, 1) == 1.25
    assert bench.replica_tok_s(1, 10, 2.0) == pytest.approx(5000.0)
