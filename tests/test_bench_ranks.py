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


def test_traffic_hash_covers_the_kernels_and_not_the_host_pipeline():
    """bench.py reports the captured DRAM traffic only while a hash of the
    tensor-core kernel sources (comments removed) matches the capture's. The
    host-buffer pipeline that closes kernels_tc.cu launches the same kernels for
    the other entry point and is left out; any change to the kernels, their
    device-buffer launches or the shared headers changes the hash."""
    csrc = os.path.join(bench.ROOT, "pair_representation_triangular_gb300", "csrc")
    src = {}
    for name in bench.TRAFFIC_SOURCES:
        with open(os.path.join(csrc, name)) as f:
            src[name] = f.read()
    base = bench.kernel_source_sha(src.__getitem__)
    assert base == bench.kernel_source_sha()

    def sha_with(name, text):
        edited = dict(src)
        edited[name] = text
        return bench.kernel_source_sha(edited.__getitem__)

    k = src["kernels_tc.cu"]
    cut = k.index(bench.HOST_PIPELINE_START)
    assert sha_with("kernels_tc.cu", k + "\nstatic int after_the_pipeline = 1;\n") == base
    assert sha_with("kernels_tc.cu", k[:cut] + k[cut:].replace("8 * wave", "6 * wave")) == base
    assert sha_with("kernels_tc.cu", "// a comment line\n" + k) == base
    kernel_line = "constexpr int BM = 128;"
    assert kernel_line in k[:cut]
    assert sha_with("kernels_tc.cu", k.replace(kernel_line, "constexpr int BM = 64;", 1)) != base
    launch = "launch_k3(t, s, map_out, 0, ntiles, false)"
    assert launch in k[:cut]
    assert sha_with("kernels_tc.cu", k.replace(launch, "launch_k3(t, s, map_out, 0, ntiles, true)", 1)) != base
    assert sha_with("tc_ptx.cuh", src["tc_ptx.cuh"] + "\n#define ANOTHER 1\n") != base
