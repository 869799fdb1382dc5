"""The N > 1 bench path on CPU: two gloo ranks agree on the slowest rank's
time, and the whole-job rate counts every rank's work over that time
(weak scaling; each GPU is an independent replica)."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    ms = [3.0, 5.5][rank]
    slowest = bench.max_over_ranks(ms, ws)
    bench.barrier(ws)
    rate = bench.job_throughput(1000.0, slowest, ws)
    out.put((rank, slowest, rate))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    for rank, slowest, rate in res:
        assert slowest == pytest.approx(5.5)
        assert rate == pytest.approx(2 * 1000.0 / 5.5e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(4.25, 1) == 4.25
    assert bench.job_throughput(10.0, 2.0, 1) == pytest.approx(5000.0)
