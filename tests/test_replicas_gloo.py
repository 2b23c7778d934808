"""The replica path of bench.py on CPU: two gloo ranks agree on the slowest rank's timings and
the whole-job figure counts both ranks' bytes (the GPU run uses the same code over NCCL)."""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q) -> None:
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        # rank r is slower on the first timing, faster on the second
        got = bench.max_over_ranks([100.0 + 10 * r, 50.0 - 5 * r, 7.0], w, torch.device("cpu"))
        q.put((r, w, lr, got))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_timings():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[:3] for o in out] == [(0, 2, 0), (1, 2, 1)]
    for o in out:
        assert o[3] == [110.0, 50.0, 7.0]


def test_whole_job_figure_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_gbps(2.0e9, 1, 1.0e6)  # 2 GB in one second
    assert one == pytest.approx(2.0)
    assert bench.whole_job_gbps(2.0e9, 4, 1.0e6) == pytest.approx(4 * one)
    assert bench.max_over_ranks([3.0, 1.0], 1, torch.device("cpu")) == [3.0, 1.0]
