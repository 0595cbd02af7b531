"""The multi-rank path of bench.py on the CPU (gloo, world size 2): the step time is the
maximum over ranks and the whole-job value counts every replica's calls.  The bench runs
one independent replica per GPU (the projection needs no exchange), so this host logic is
all there is to the N > 1 path."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step_ms = [5.0, 7.5][rank]                       # rank 1 is the slow replica
        worst = bench.max_over_ranks(step_ms, torch.device("cpu"))
        ws, r, local = bench.dist_env()
        q.put((rank, worst, bench.job_us_per_call(worst, 1000, world), (ws, r, local)))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_on_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst, job_us, env in got:
        assert worst == 7.5                              # the slowest rank sets the step time
        assert job_us == pytest.approx(7.5 * 1000.0 / (1000 * 2))   # 2000 calls in 7.5 ms
        assert env == (2, rank, rank)


def test_single_rank_value_is_the_per_call_time():
    assert bench.job_us_per_call(5.45, 1000, 1) == pytest.approx(5.45)
