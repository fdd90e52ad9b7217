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
    shapes = src["tc_shapes.h"]
    kernel_line = "constexpr int BM = 128;"
    assert kernel_line in shapes
    assert sha_with("tc_shapes.h", shapes.replace(kernel_line, "constexpr int BM = 64;", 1)) != base
    k2 = src["tc_k2.cu"]
    assert sha_with("tc_k2.cu", k2.replace("SPS == SPS - 1", "SPS == 0", 1)) != base
    launch = "launch_k3(t, s, map_out, 0, ntiles, false)"
    assert launch in k[:cut]
    assert sha_with("kernels_tc.cu", k.replace(launch, "launch_k3(t, s, map_out, 0, ntiles, true)", 1)) != base
    assert sha_with("tc_ptx.cuh", src["tc_ptx.cuh"] + "\n#define ANOTHER 1\n") != base


def _run_bench(args, env=None, timeout=240):
    import subprocess
    import sys
    full_env = dict(os.environ)
    full_env.update(env or {})
    return subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=timeout, env=full_env)


def test_reference_arm_prints_one_contract_line():
    """--impl reference times the CPU oracle on this host and prints exactly one
    JSON line with the native arm's metric, unit and config, the oracle's own
    cpu_baseline and an e2e block with no host<->device bytes. A step is one
    bounded sample: ms_per_step is its measured wall time (so steps x
    ms_per_step is the work the arm did), and at this tiny size the sample
    covers every row, so it is one whole forward and value = cells / time."""
    import json
    r = _run_bench(["--impl", "reference", "--workload", "b2-n32-d64-h4-f32",
                    "--steps", "2", "--warmup", "1"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    assert rec["metric"] == bench.METRIC and rec["unit"] == "pair-cells/s"
    assert rec["value"] > 0 and rec["higher_is_better"] is True
    assert (rec["n_gpus"], rec["steps"], rec["warmup"]) == (1, 2, 1)
    assert rec["step"].startswith("one bounded sample")
    assert rec["ms_per_step"] == pytest.approx(2 * 32 * 32 / rec["value"] * 1e3, rel=1e-3)
    assert rec["config"]["workload"] == "b2-n32-d64-h4-f32"
    cb = rec["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == rec["value"]
    assert "rows" in cb["sample"]
    assert rec["e2e"] == {"value": rec["value"], "unit": "pair-cells/s",
                          "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    """Under torchrun only rank 0 runs the reference arm; the others exit 0
    without output or work."""
    r = _run_bench(["--impl", "reference", "--workload", "b2-n32-d64-h4-f32",
                    "--steps", "1", "--warmup", "0"], env={"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_clock_summary_reports_median_and_throttle_reasons():
    """The sampler's rows are nvidia-smi CSV fields (index, clocks.sm,
    clocks.max.sm, power, active mask, hw_slowdown, hw_thermal_slowdown,
    sw_thermal_slowdown, sw_power_cap); the summary gives the median SM clock,
    the maximum clock and every throttle reason seen Active at least once."""
    clk = bench.ClockSampler(0)
    assert clk.summary()["reasons"] == ["clock sampling unavailable"]
    idle = ["Not Active"] * 4
    clk.rows = [["0", "2070", "2070", "700.1", "0x0", *idle],
                ["0", "1980", "2070", "1390.0", "0x4", "Not Active", "Not Active", "Not Active",
                 "Active"],
                ["0", "2070", "2070", "900.0", "0x0", *idle],
                ["0", "[N/A]", "2070", "900.0", "0x0", *idle]]
    s = clk.summary()
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 4
    clk.rows.append(["0", "1500", "2070", "800.0", "0x8", "Active", "Not Active", "Active",
                     "Not Active"])
    assert clk.summary()["reasons"] == ["sw_power_cap", "hw_slowdown", "sw_thermal_slowdown"]


def test_algorithmic_work_matches_the_per_cell_figures(monkeypatch):
    """The roofline's algorithmic work per cell at the N = 768 bf16 workload:
    K1 reads x and writes q, k, v, g and the fp32 bias (2D + 8D + 4h = 1296 B);
    bias_rows reads that plane and writes the fp16 one (6h = 24 B); K2 reads
    q, k, v and the fp16 bias and writes o (6D + 2h + 2D = 1032 B) plus the mask
    bit rows, for 4 B N^3 D FLOPs; K3 reads g and o and writes out (768 B); the
    mask summary reads the int32 mask. The captured traffic is reported only
    while the kernel sources hash to the capture's."""
    from pair_representation_triangular_gb300 import workloads as W
    w = W.WORKLOADS["b1-n768-d128-h4-bf16-pad700"]
    P, N, D, h = w.cells, w.N, w.D, w.h
    work = bench.algorithmic_work(w)
    bits = N * (1 + 8 * ((N + 63) // 64))
    assert work["ln_proj"]["bytes"] == 1296 * P
    assert work["bias_rows"]["bytes"] == 24 * P
    assert work["ln_proj"]["flops"] == 2.0 * P * D * (4 * D + h)
    assert work["row_attn"]["bytes"] == 1032 * P + bits
    assert work["row_attn"]["flops"] == 4.0 * N ** 3 * D
    assert work["gate_out"]["bytes"] == 768 * P
    assert work["mask_summary"]["bytes"] == 4 * P + bits
    assert work["row_attn"]["flops"] / 1e9 == pytest.approx(231.9, abs=0.1)
    assert bench.measured_traffic("row_attn_tc", P) == pytest.approx(
        bench.TRAFFIC_PER_CELL["row_attn_tc"] * P)
    monkeypatch.setitem(bench.TRAFFIC_PER_CELL, "source_sha256", "0" * 16)
    assert bench.measured_traffic("row_attn_tc", P) is None
