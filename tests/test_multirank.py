"""The multi-GPU path of bench.py is independent replicas: each rank times its
own step and rank 0 reports the slowest rank's time.  These tests run that
reduction with two gloo ranks on the CPU (no GPU involved)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r is slower on the first value, faster on the second
    got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5], world)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got))


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results[0] == results[1] == [2.0, 10.0, 0.5]


def test_single_process_is_identity_and_value_is_weak_scaling():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
    # 4 ranks, each 1e12 FLOP per step, slowest step 2 ms -> 2000 TFLOP/s
    assert bench.whole_job_value(1e12, 4, 2.0, 1e12) == pytest.approx(2000.0)
