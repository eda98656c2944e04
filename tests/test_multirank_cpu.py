"""The multi-rank bench logic on CPU with the gloo backend (world size 2).

Rows are independent, so N ranks each select their own batch and the job's
time is the slowest rank's; bench.py takes the maximum over ranks with one
all-reduce and reports ranks x rows x steps over that time.  Here two CPU
processes stand in for two GPUs: each reports a different local time and
both must come back with the maximum and the same job rate.  No GPU, no
CUDA call.
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


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        env = bench.dist_env()
        local_ms = 100.0 + 25.0 * rank          # rank 1 is the slower one
        t = bench.max_over_ranks(local_ms, ws, torch.device("cpu"))
        rate = bench.job_rows_per_s(ws, 8192, 20, t)
        q.put((rank, env, t, rate))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ps = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in ps:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(ws))
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, t, rate in got:
        assert env == (ws, rank, rank)
        assert t == 125.0
        assert rate == pytest.approx(2 * 8192 * 20 / 0.125)


def test_one_rank_is_a_no_op():
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.job_rows_per_s(1, 100, 10, 1000.0) == pytest.approx(1000.0)
