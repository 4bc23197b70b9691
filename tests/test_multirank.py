"""The multi-GPU arm of the benchmark is replicas only: every rank runs its own
cache with no collective on the data path, and the job's throughput is all
ranks' units over the slowest rank's time.  This checks that host logic with
two gloo ranks on the CPU (no GPU): the time reduction takes the maximum over
ranks and the whole-job value counts every rank's work.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [10.0 + 5.0 * rank, 30.0 - 10.0 * rank, 0.0]  # rank 0: 10, 30; rank 1: 15, 20
        reduced = bench.max_over_ranks(local, world, "cpu")
        out[rank] = reduced + [bench.whole_job_value(1e9, world, reduced[0], 1e-9)]
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        got = dict(out)
    for rank in (0, 1):
        ms, e2e_ms, graph_ms, value = got[rank]
        assert (ms, e2e_ms, graph_ms) == (15.0, 30.0, 0.0)  # max over ranks, per timing
        assert value == pytest.approx(2 * 1e9 * 1e-9 / 15e-3)  # both replicas' work over the slowest time


def test_single_rank_is_untouched():
    assert bench.max_over_ranks([1.5, 2.5], 1, "cpu") == [1.5, 2.5]
    assert bench.whole_job_value(5e9, 1, 2.0, 1e-9) == pytest.approx(2500.0)
