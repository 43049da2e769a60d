"""The multi-rank path of bench.py on CPU: two gloo ranks (127.0.0.1), the
slowest rank's time and the whole-job value of independent replicas."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        local_ms = [120.0, 150.0][rank]  # rank 1 is the slow one
        total = bench.max_over_ranks(local_ms, torch.device("cpu"))
        out[rank] = (total, bench.replicas_value(1_000_000, 10, world, total))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1]
    total, value = out[0]
    assert total == 150.0
    # 2 ranks x 10 steps x 1 MB over 150 ms
    assert abs(value - 2 * 10 * 1_000_000 / 0.150 / 1e9) < 1e-12


def test_single_process_is_its_own_max():
    import bench
    assert bench.max_over_ranks(7.5, torch.device("cpu")) == 7.5
