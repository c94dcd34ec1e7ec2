"""The cross-rank host logic of bench.py, world size 2 over gloo on CPU.

The path has no exchange step (output rows are independent), so N GPUs run
N replicas. The only cross-rank logic is the whole-job time (the maximum over
ranks, after a barrier) and the whole-job value (every rank's bytes over that
time). Both are checked here without a GPU.
"""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        dist.barrier()
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        t = bench.job_time_ms(torch, local_ms, w, torch.device("cpu"))
        v = bench.job_value(w, 2.0e9, t / 4)  # 2 GB per rank and step, 4 steps
        out.put((r, w, local, t, v))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_sum_the_bytes():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out))
             for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(out.get(timeout=180) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, (r, w, local, t, v) in enumerate(res):
        assert (r, w, local) == (rank, 2, rank)
        assert t == 15.0                       # max over ranks, on both
        # 2 ranks x 2 GB per step in 15 ms / 4 per step
        assert v == pytest.approx(2 * 2.0e9 / (15.0e-3 / 4) / 1e9)


def test_one_rank_keeps_its_own_time():
    assert bench.job_time_ms(torch, 12.5, 1, torch.device("cpu")) == 12.5
    assert bench.job_value(1, 1.0e9, 1.0) == pytest.approx(1000.0)
