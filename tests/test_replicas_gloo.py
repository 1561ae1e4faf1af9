"""The N > 1 path of bench.py on CPU: two gloo ranks, each timing its own
replica; the job's step time is the max over ranks and the value sums the
replicas' work (weak scaling, no collective on the data path)."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [12.5, 20.0][rank]
    worst = bench.max_over_ranks(local_ms)
    value = bench.step_value(0.001, world, worst)
    out[rank] = (worst, value)
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1]
    worst, value = out[0]
    assert worst == 20.0
    # 2 replicas x 1 ms of roofline work in a 20 ms step = 10 %
    assert value == pytest.approx(10.0)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.step_value(0.5e-3, 1, 1.0) == pytest.approx(50.0)
