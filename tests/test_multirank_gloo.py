"""The N > 1 host logic of the benchmark, on CPU with gloo, world size 2.

Rows are independent, so the multi-GPU path is replicas with no data-path
exchange: each rank runs its own batch, and the only collectives are the
barrier around the timed region and the max over ranks of the elapsed time.
These tests run that reduction and the whole-job rate on two gloo ranks."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, times: list, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    dist.barrier()
    mx = bench.max_over_ranks(times[rank], world)
    rate = bench.whole_job_rate(256, 10, world, mx)
    out.put((rank, mx, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_rate_on_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [0.5, 0.8]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, rate in res:
        assert mx == pytest.approx(0.8)
        assert rate == pytest.approx(256 * 10 * 2 / 0.8)


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.whole_job_rate(256, 4, 1, 2.0) == 512.0
