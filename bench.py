"""Benchmark: forward passes of triangular self-attention (starting node, or the
ending node with --node ending) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--node starting|ending] [--mask-mode 0|1] [--impl reference]

One step is one full forward pass (LayerNorm + projections, row attention, gate +
output projection) over one batch of seeded synthetic input, the default being
the B=1, N=768, D=128, h=4 bf16 workload with a padded-sequence mask (700 of 768
residues kept). Prints one JSON line (rank 0).

value      pair-cells/s = B*N^2 / (device time per forward), inputs resident in
           HBM, L2 flushed (256 MB write) before every timed step.
e2e        the same metric through tri_attn_forward_host: pinned host buffers
           (filled once) are reused; every step copies pair_repr and pair_mask
           host->device and the output device->host inside the timed region.
roofline   the dominant kernel (largest share of device time) against its
           algorithmic bytes or FLOPs per launch.
cpu_baseline  the CPU oracle (fp64 numpy) on a bounded sample of the same
           workload, timed on this host's cores.

--impl reference times the CPU oracle alone (the reference arm of this
benchmark) and prints the same JSON line with "impl": "reference".
Under torchrun every rank runs its own independent forward passes (weak
scaling over independent problems, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "b1-n768-d128-h4-bf16-pad700"
METRIC = "pair-cells/s per forward (B*N^2/s)"
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--mask-mode", type=int, default=0)
    ap.add_argument("--node", default="starting", choices=["starting", "ending"])
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    return ap.parse_args()


# ------------------------------------------------------------------ workload math
def algorithmic_work(w):
    """Per-kernel algorithmic FLOPs and HBM bytes of one forward, each tensor
    read or written once: K1 reads x and writes q, k, v, g and the fp32 bias
    plane; on the bf16 path bias_rows reads that plane and writes the fp16 one
    the attention reads (fp32 on the fp32 path); the mask summary reads the
    int32 mask and writes its bit rows and row flags; K2 reads q, k, v, the bias
    plane and the bit rows, writes o; K3 reads g and o, writes out."""
    P, D, h, N, B = w.cells, w.D, w.h, w.N, w.B
    s = 2 if w.dtype == "bf16" else 4
    bias32 = 4 * P * h
    bias_k2 = (2 if w.dtype == "bf16" else 4) * P * h
    bits = B * N * (1 + 8 * ((N + 63) // 64))
    return {
        "ln_proj": {"flops": 2.0 * P * D * (4 * D + h),
                    "bytes": P * D * s + 4 * P * D * s + bias32},
        "bias_rows": {"flops": 0.0, "bytes": bias32 + 2 * P * h},
        "row_attn": {"flops": 4.0 * B * N ** 3 * D,
                     "bytes": 3 * P * D * s + bias_k2 + bits + P * D * s},
        "gate_out": {"flops": 2.0 * P * D * D, "bytes": 3 * P * D * s},
        "mask_summary": {"flops": 0.0, "bytes": 4 * P + bits},
    }


# DRAM traffic per pair cell (dram__bytes_read.sum + dram__bytes_write.sum of
# one launch, divided by its B*N^2 cells) from an ncu capture of the B=1,
# N=384 bf16 workload (the N = 768 workload is too large to capture whole).
# It holds for the tensor-core kernel code whose SHA-256 prefix (comments
# removed) is recorded here; for any other code the bench reports traffic as
# null.
TRAFFIC_SOURCES = ("kernels_tc.cu", "tc_k1.cu", "tc_k2.cu", "tc_k3.cu", "tc_kernels.cuh",
                   "tc_device.cuh", "tc_shapes.h", "tc_ptx.cuh", "common.cuh")
# The host-buffer pipeline closes kernels_tc.cu: it launches the same kernels
# for the host-buffer entry point and leaves the device-buffer forward that the
# capture measured unchanged, so the hash stops where it begins.
HOST_PIPELINE_START = "cudaError_t tri_tc_forward_host("
TRAFFIC_PER_CELL = {
    "source_sha256": "fa1ded6d28865fbe",
    "capture": "b1-n384-d128-h4-bf16-pad320",
    "ln_proj_tc": (37.937408e6 + 97.383168e6) / 147456,
    "row_attn_tc": (104.302080e6 + 12.538880e6) / 147456,
    "gate_out_tc": (75.562496e6 + 2.213632e6) / 147456,
    "bias_rows": (2.376960e6 + 0.000000e6) / 147456,
}


def code_lines(text: str) -> str:
    """Source text without // comments, trailing blanks and empty lines, so that
    a change of comments keeps the hash of the code."""
    out = []
    for line in text.splitlines():
        line = line.split("//", 1)[0].rstrip()
        if line:
            out.append(line)
    return "\n".join(out)


def kernel_source_sha(read=None) -> str:
    import hashlib
    h = hashlib.sha256()
    for name in TRAFFIC_SOURCES:
        if read is None:
            with open(os.path.join(ROOT, "pair_representation_triangular_gb300", "csrc", name)) as f:
                text = f.read()
        else:
            text = read(name)
        if name == "kernels_tc.cu" and HOST_PIPELINE_START in text:
            text = text[:text.index(HOST_PIPELINE_START)]
        h.update(code_lines(text).encode())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, cells: int):
    """Bytes one launch of `kernel` moves to and from DRAM, scaled by cells from
    the recorded capture, or None if the kernel sources changed since."""
    per_cell = TRAFFIC_PER_CELL.get(kernel)
    if per_cell is None or kernel_source_sha() != TRAFFIC_PER_CELL["source_sha256"]:
        return None
    return per_cell * cells


def max_over_ranks(x: float, device) -> float:
    """Largest value of x over all ranks of the default process group (x itself
    when no group is initialised or it has one rank)."""
    import torch
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return x
    if torch.distributed.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(cells_per_rank: int, world: int, ms_per_step: float) -> float:
    """Pair-cells per second over all ranks: every rank runs its own forward of
    `cells_per_rank` cells per step, and the slowest rank's step time counts."""
    return world * cells_per_rank / (ms_per_step / 1e3)


def kernel_key(name: str) -> str:
    for k in ("ln_proj", "bias_rows", "row_attn", "gate_out", "mask_summary"):
        if name.startswith(k):
            return k
    return name


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons every 25 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        sm = [float(r[1]) for r in self.rows if len(r) > 2 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) > 2 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = []
        for r in self.rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active" and n not in reasons:
                    reasons.append(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


# ------------------------------------------------------------------ CPU oracle baseline
def _oracle_rows_worker(args):
    """Softmax lines of the oracle forward in a spawned worker (single-threaded
    BLAS): rows i of the grid for the starting node, columns for the ending
    node."""
    x_lines, mask, params, h, lines, mode, bias_b, ending = args
    import numpy as np
    import oracle.tri_attn_oracle as O
    P = {k: np.asarray(v, np.float64) for k, v in params.items()}
    out = []
    for n, (b, a) in enumerate(lines):
        x_hat = O.layer_norm(np.asarray(x_lines[n], np.float64), P["gamma"], P["beta"])
        q, k, v, g, _ = O.project(x_hat, P)
        if ending:
            keep, bias_l = O.column_keep(mask, b, a, mode), O.column_bias(bias_b)
        else:
            keep, bias_l = O.keep_matrix(mask, b, a, mode), bias_b
        o = O.row_attention(q, k, v, bias_l, keep, h)
        out.append(O.output_projection(g, o, P))
    return len(out)


def _oracle_bias_worker(args):
    x_cells, params, = args
    import numpy as np
    import oracle.tri_attn_oracle as O
    P = {k: np.asarray(v, np.float64) for k, v in params.items()}
    x_hat = O.layer_norm(np.asarray(x_cells, np.float64), P["gamma"], P["beta"])
    return O.linear(x_hat, P["Wb"])


def cpu_oracle_sample(w, inp, mode, budget_s=20.0, cores=None, ending=False):
    """Time the oracle on this host: the full bias plane (every cell) plus as many
    softmax lines (rows, or columns for the ending node) as fit in about
    `budget_s`, spread over `cores` spawned processes; the full-forward time is
    extrapolated from the per-line time. Returns the JSON object of the
    baseline."""
    import numpy as np
    cores = cores or os.cpu_count() or 1
    env_keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in env_keys}
    for k in env_keys:
        os.environ[k] = "1"
    ctx = mp.get_context("spawn")
    B, N = w.B, w.N
    try:
        with ctx.Pool(cores) as pool:
            t0 = time.perf_counter()
            xs = inp["x"].reshape(B * N, N, w.D)
            parts = pool.map(_oracle_bias_worker, [(xs[r], inp["params"]) for r in range(B * N)],
                             chunksize=max(1, (B * N) // (4 * cores)))
            bias = np.stack(parts).reshape(B, N, N, w.h).transpose(0, 3, 1, 2)
            t_bias = time.perf_counter() - t0
            # rows: one per worker first to measure, then as many as the budget allows
            rows_all = [(b, i) for b in range(B) for i in range(N)]
            done = 0
            t_rows = 0.0
            batch = cores
            while done < len(rows_all):
                chunk = rows_all[done:done + batch]
                jobs = [(((inp["x"][b, :, i] if ending else inp["x"][b, i]),), inp["pair_mask"],
                         inp["params"], w.h, [(b, i)], mode, bias[b], ending) for b, i in chunk]
                t1 = time.perf_counter()
                pool.map(_oracle_rows_worker, jobs, chunksize=1)
                t_rows += time.perf_counter() - t1
                done += len(chunk)
                if t_bias + t_rows > budget_s:
                    break
                batch = min(len(rows_all) - done, max(cores, int(done * (budget_s - t_bias - t_rows)
                                                                  / max(t_rows, 1e-9) * 0.5)))
                batch = max(batch, 1)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    t_full = t_bias + t_rows * (len(rows_all) / done)
    value = B * N * N / t_full
    return {"value": value, "unit": "pair-cells/s", "cores": cores, "kind": "oracle",
            "sample_s": t_bias + t_rows,
            "sample": (f"fp64 numpy oracle, {cores} spawned single-thread processes: full bias "
                       f"plane ({B * N * N} cells, {t_bias:.2f} s) + {done} of {len(rows_all)} "
                       f"rows ({t_rows:.2f} s); full-forward time extrapolated linearly "
                       f"in rows: {t_full:.1f} s")}


def bench_config(w, args, world):
    """The `config` object of both arms' JSON lines."""
    return {"workload": w.name, "B": w.B, "N": w.N, "D": w.D, "h": w.h,
            "node": args.node,
            "mask_mode": "row-key" if args.mask_mode == 0 else "query-key",
            "l2": f"flushed (256 MB write) before each timed step; x is "
                  f"{w.cells * w.D * (2 if w.dtype == 'bf16' else 4) / 1e6:.0f} MB",
            "parallelism": f"{world} independent problems, one per GPU"}


# ------------------------------------------------------------------ native arm
def run_native(args, rank, world):
    import numpy as np
    import torch
    from pair_representation_triangular_gb300 import binding as tb
    from pair_representation_triangular_gb300 import build as tbuild
    from pair_representation_triangular_gb300 import workloads as W

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    tbuild.build()
    tb.load_library()
    w = W.WORKLOADS[args.workload]
    inp = W.make_inputs(w)
    td = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dt = tb.TRI_ATTN_BF16 if w.dtype == "bf16" else tb.TRI_ATTN_F32
    params = {k: torch.from_numpy(v).to(dev, td) for k, v in inp["params"].items()}
    x = torch.from_numpy(inp["x"]).to(dev, td)
    m = torch.from_numpy(inp["pair_mask"]).to(dev)
    out = torch.empty_like(x)
    node = tb.TRI_ATTN_ENDING_NODE if args.node == "ending" else tb.TRI_ATTN_STARTING_NODE
    mod = tb.TriangularAttention(w.B, w.N, w.D, w.h, dt, args.mask_mode | node, params)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        mod.forward(x, m, out)
    st = mod.sync_check()
    if st != tb.TRI_ATTN_OK:
        raise RuntimeError(f"warm-up forward failed: {tb.tri_attn_status_string(st)}")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        # Keep the GPU under load until the sampler reports (at most ~2 s), so
        # that its samples cover the loaded clocks around the timed steps.
        t_wait = time.perf_counter()
        while clk.proc is not None and len(clk.rows) < 2 and time.perf_counter() - t_wait < 2.0:
            mod.forward(x, m, out)
            torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        for s in range(args.steps):
            flush.fill_(float(s))                       # evict L2 (outside the timed pair)
            ev[s][0].record(stream)
            mod.forward(x, m, out)
            ev[s][1].record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    st = mod.sync_check()
    if st != tb.TRI_ATTN_OK:
        raise RuntimeError(f"timed forward failed: {tb.tri_attn_status_string(st)}")
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_total = max_over_ranks(sum(step_ms), dev)
    ms_per_step = ms_total / args.steps
    value = whole_job_rate(w.cells, world, ms_per_step)

    # Per-kernel breakdown: the same steps again with the library's CUDA events
    # between the kernels (kept out of the headline pass above).
    tb.tri_attn_enable_kernel_timing(mod.handle, True)
    kernel_ms = {}
    per_forward = 0
    for s in range(args.steps):
        flush.fill_(float(s))
        mod.forward(x, m, out)
        times = tb.tri_attn_kernel_times(mod.handle)
        per_forward = len(times)
        for name, ms in times:
            kernel_ms.setdefault(name, []).append(ms)
    tb.tri_attn_enable_kernel_timing(mod.handle, False)
    launches = per_forward * args.steps                 # kernels in the timed pass

    # e2e: host buffers through the C ABI (copies inside the timed region)
    xh = torch.from_numpy(inp["x"]).to(td).pin_memory()
    mh = torch.from_numpy(inp["pair_mask"]).pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    mod.forward_host(xh, mh, oh)
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        mod.forward_host(xh, mh, oh)
    e2e_s = max_over_ranks((time.perf_counter() - t0) / args.e2e_steps, dev)
    h2d = xh.numel() * xh.element_size() + mh.numel() * mh.element_size()
    d2h = oh.numel() * oh.element_size()

    # roofline of the dominant kernel
    work = algorithmic_work(w)
    avg = {k: sum(v) / len(v) for k, v in kernel_ms.items()}
    total = sum(avg.values())
    top = max(avg, key=avg.get)
    kw = work[kernel_key(top)]
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
        peak_src = "measured"
    except OSError:
        peak_src = "fallback"
    hbm = peaks.get("hbm_gbs", 6800.0)
    if w.dtype == "bf16":
        tflops, fbound = peaks.get("bf16_tflops", 1900.0), "tensor"
    else:
        # fp32 FFMA path: SMs x 128 fp32 lanes x 2 FLOP per FMA x the maximum SM clock
        sm_mhz = clk.summary().get("sm_max_mhz") or 2070.0
        tflops = torch.cuda.get_device_properties(dev).multi_processor_count * 128 * 2 * sm_mhz / 1e6
        fbound = "alu"
    t_s = avg[top] / 1e3
    t_bytes = kw["bytes"] / (hbm * 1e9)
    t_flops = kw["flops"] / (tflops * 1e12)
    if t_flops >= t_bytes:
        roof = {"bound": fbound, "achieved": kw["flops"] / t_s / 1e12, "peak": tflops,
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": kw["bytes"] / t_s / 1e9, "peak": hbm, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = top
    if kernel_key(top) == "row_attn" and w.dtype == "bf16":
        # The attention kernel's three floors: tensor FLOPs, HBM bytes and the
        # special-function unit's exp2 rate (one exp2 per line, head, query and
        # key; 32 per clock per SM as measured on this GPU, at the maximum clock).
        sm_mhz = clk.summary().get("sm_max_mhz") or 2070.0
        sfu_rate = torch.cuda.get_device_properties(dev).multi_processor_count * 32 * sm_mhz * 1e6
        t_sfu = w.B * w.h * w.N ** 3 / sfu_rate
        roof["floors_ms"] = {"tensor": round(t_flops * 1e3, 4), "hbm": round(t_bytes * 1e3, 4),
                             "sfu": round(t_sfu * 1e3, 4)}
        roof["sfu_frac"] = round(t_sfu / t_s, 4)
    roof["peak_source"] = (peak_src + " (burst)" if fbound == "tensor" or t_bytes > t_flops
                           else "derived: SMs x 128 FFMA lanes x 2 x max SM clock")
    roof["traffic"] = measured_traffic(top, w.cells) if w.dtype == "bf16" else None
    if roof["traffic"] is not None:
        roof["traffic_note"] = ("dram read+write bytes per launch, scaled by cells from the ncu "
                                "capture of " + TRAFFIC_PER_CELL["capture"])
    roof["kernel_ms"] = {k: round(v, 5) for k, v in avg.items()}
    roof["kernel_share"] = {k: round(v / total, 4) for k, v in avg.items()}
    roof["kernel_roofline_frac"] = {}
    for k, v in avg.items():
        kk = work[kernel_key(k)]
        t_roof = max(kk["bytes"] / (hbm * 1e9), kk["flops"] / (tflops * 1e12))
        roof["kernel_roofline_frac"][k] = round(t_roof / (v / 1e3), 4)

    result = {
        "metric": METRIC, "value": value, "unit": "pair-cells/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic (seeded)",
        "config": bench_config(w, args, world),
        "e2e": {"value": world * w.cells / e2e_s, "unit": "pair-cells/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "roofline": roof,
        "clocks": clk.summary(),
    }
    mod.close()
    return result, w, inp


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        from pair_representation_triangular_gb300 import workloads as W
        w = W.WORKLOADS[args.workload]
        inp = W.make_inputs(w)
        # One step of this arm is one bounded sample of the forward (the whole
        # bias plane and as many softmax lines as fit its time budget); `value`
        # is the whole-forward rate extrapolated from it, `ms_per_step` the
        # sample's measured wall time, so steps x ms_per_step is the work done.
        vals, secs = [], []
        base = None
        for s in range(args.warmup + args.steps):
            budget = 2.0 if s < args.warmup else max(2.0, 150.0 / max(args.steps, 1))
            r = cpu_oracle_sample(w, inp, args.mask_mode, budget_s=budget,
                                  ending=args.node == "ending")
            if s >= args.warmup:
                vals.append(w.cells / r["value"])      # extrapolated whole-forward seconds
                secs.append(r["sample_s"])
                base = r
        value = w.cells / statistics.mean(vals)
        base["value"] = value
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": value, "unit": "pair-cells/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": statistics.mean(secs) * 1e3,
            "step": "one bounded sample of the forward; value extrapolates it to a whole forward",
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": bench_config(w, args, world),
            "cpu_baseline": base,
            "e2e": {"value": value, "unit": "pair-cells/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }))
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    result, w, inp = run_native(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            result["cpu_baseline"] = cpu_oracle_sample(w, inp, args.mask_mode, budget_s=20.0,
                                                       ending=args.node == "ending")
        print(json.dumps(result))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
