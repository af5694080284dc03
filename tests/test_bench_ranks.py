"""Multi-rank host logic of bench.py on CPU: two gloo ranks, each an independent
replica; the job's step time is the maximum over ranks and its throughput counts
the tokens of every rank."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = bench.dist_info()
        ms_all, value = bench.job_throughput(1.0 + 0.5 * r, 53, w, "cpu")
        q.put((r, w, ms_all, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time_and_sum_tokens():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, w, ms_all, value) in enumerate(out):
        assert rank == r and w == world
        assert ms_all == pytest.approx(1.5)                 # the slower rank's time
        assert value == pytest.approx(2 * 53 / 1.5e-3)      # tokens of both ranks / that time


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    ms_all, value = bench.job_throughput(2.0, 64, 1, "cpu")
    assert ms_all == 2.0 and value == pytest.approx(64 / 2e-3)
