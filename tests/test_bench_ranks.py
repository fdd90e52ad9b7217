"""Host logic of the multi-rank benchmark on CPU: two gloo ranks (127.0.0.1)
take the slowest rank's time and report the whole-job rate. Under torchrun
every rank runs its own independent forward passes, so the only exchange is
this max-reduction of the measured times."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank                     # rank 1 is the slower one
        ms = bench.max_over_ranks(local_ms, "cpu")
        out[rank] = (ms, bench.whole_job_rate(1000, world, ms))
    finally:
        torch.distributed.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, rate = res[rank]
        assert ms == pytest.approx(15.0)
        assert rate == pytest.approx(2 * 1000 / 0.015)


def test_single_process_is_unchanged():
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.whole_job_rate(589824, 1, 1.0) == pytest.approx(589824e3)
