"""The bench's multi-rank plumbing on CPU (gloo, world_size 2).

Each rank runs an independent replica of the layer ("replicas only": the layer
has no cross-GPU step), so the only collective is the timing reduction: the
whole-job throughput divides every rank's tokens by the slowest rank's time.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = [2.0, 3.5][rank]
    e2e = [4.0, 1.0][rank]
    got = bench.reduce_max([ms, e2e])
    q.put((rank, got, bench.job_throughput(world, 4096, got[0])))
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_max_and_job_throughput_gloo_two_ranks():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, tput in out:
        assert got == [3.5, 4.0]                              # max over ranks, per quantity
        assert tput == pytest.approx(2 * 4096 / 3.5e-3)       # all ranks' tokens / slowest time


def test_single_process_is_identity():
    import bench

    assert not dist.is_initialized()
    assert bench.reduce_max([1.5, 2.5]) == [1.5, 2.5]
    assert bench.job_throughput(1, 4096, 0.2) == pytest.approx(4096 / 0.2e-3)
