"""The N > 1 host logic of bench.py on CPU: two gloo ranks, the job time is the
slowest rank's and the value counts every rank's units (weak scaling,
replicas only: the scan has no data-path exchange between GPUs)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r took (r + 1) * 100 ms for 10 steps, forward (r + 1) * 40 ms
    ms, value, fwd_value = bench.aggregate((rank + 1) * 100.0, (rank + 1) * 40.0, world, 8 * 1024, 10)
    q.put((rank, ms, value, fwd_value))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value, fwd_value in out:
        assert ms == pytest.approx(20.0)  # the slower rank: 200 ms / 10 steps
        assert value == pytest.approx(2 * 8 * 1024 / 0.020)
        assert fwd_value == pytest.approx(2 * 8 * 1024 / 0.008)


def test_single_rank_needs_no_process_group():
    import bench
    ms, value, fwd_value = bench.aggregate(50.0, 20.0, 1, 100, 5)
    assert ms == pytest.approx(10.0)
    assert value == pytest.approx(100 / 0.010)
    assert fwd_value == pytest.approx(100 / 0.004)
