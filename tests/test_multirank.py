"""The replicas path of bench.py on CPU: two gloo ranks agree on the
slowest rank's time and report the whole-job rate from it."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 2.0 + rank                      # rank 1 is the slow one
    slow = bench.slowest_ms(ms, dist, device="cpu")
    rate = bench.job_rate(1000.0, world, slow)
    out[rank] = (slow, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 3.0
    assert res[0][1] == res[1][1] == pytest.approx(2 * 1000.0 / 3e-3)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_ms(1.5, None) == 1.5
    assert bench.job_rate(10.0, 1, 2.0) == pytest.approx(5000.0)
