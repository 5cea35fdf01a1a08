"""Replica scaling logic of bench.py on two gloo ranks (CPU).

The decode units need no exchange, so N GPUs run N replicas; the only
cross-rank steps are the barrier and the max over ranks of the step time.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [0.5, 0.8][rank]
    dist.barrier()
    ms_max = bench.reduce_max(ms, dist, "cpu")
    gbs = bench.job_gbs(1e9, world, ms_max)
    q.put((rank, ms_max, gbs))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, gbs in res:
        assert ms_max == pytest.approx(0.8)
        assert gbs == pytest.approx(2 * 1e9 / 0.8e-3 / 1e9)


def test_single_process_identity():
    import bench
    assert bench.reduce_max(1.25) == 1.25
    assert bench.job_gbs(2e9, 1, 1.0) == pytest.approx(2000.0)
