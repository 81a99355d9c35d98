"""The multi-GPU path of bench.py is replicas only (each rank runs the whole request; no data-path
collective).  Its cross-rank bookkeeping -- slowest-rank time and whole-job throughput -- runs
here on two CPU ranks over gloo."""
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


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = 40.0 + 5.0 * rank  # rank 1 is the slower replica
    job = bench.max_over_ranks(ms, world)
    value = bench.job_throughput(6.89e13, world, job)
    dist.barrier()
    q.put((rank, job, value))
    dist.destroy_process_group()


def test_two_cpu_replicas_report_the_slowest_rank_and_whole_job_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, job, value in res:
        assert job == 45.0
        assert value == pytest.approx(2 * 6.89e13 / 0.045 / 1e12)


def test_single_rank_is_unchanged():
    import bench

    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.job_throughput(1e12, 1, 1000.0) == pytest.approx(1.0)
