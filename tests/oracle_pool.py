"""The CPU oracle over every softmax line of a workload, spread over spawned
worker processes (test infrastructure: the oracle's own functions do the
arithmetic; this module only splits the lines and gathers the results).

Each worker regenerates the workload's seeded inputs itself (cheaper than
sending 0.3 GB to every process) and evaluates its share of the lines with
``forward_rows`` (grid rows, starting node) or ``forward_ending_columns``
(grid columns, ending node). Workers are started with ``spawn``: a process
forked after the parent has touched the GPU can hang."""
import multiprocessing as mp
import os

import numpy as np


def _lines_worker(args):
    w, mode, ending, lines, edit = args
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    import oracle.tri_attn_oracle as O
    from pair_representation_triangular_gb300 import workloads as W
    inp = W.make_inputs(w)
    if edit is not None:
        edit(inp)
    if ending:
        return O.forward_ending_columns(inp["x"], inp["pair_mask"], inp["params"], w.h, lines, mode)
    return O.forward_rows(inp["x"], inp["pair_mask"], inp["params"], w.h, lines, mode)


def oracle_forward(w, mode, ending=False, procs=None, edit=None):
    """The oracle's full output (B, N, N, D), float64. `edit`, if given, is a
    picklable function applied to the regenerated inputs in every worker."""
    lines = [(b, a) for b in range(w.B) for a in range(w.N)]
    procs = max(1, min(len(lines), procs or os.cpu_count() or 1))
    shares = [lines[k::procs] for k in range(procs)]
    with mp.get_context("spawn").Pool(procs) as pool:
        parts = pool.map(_lines_worker, [(w, mode, ending, sh, edit) for sh in shares])
    out = np.empty((w.B, w.N, w.N, w.D))
    for share, part in zip(shares, parts):
        for n, (b, a) in enumerate(share):
            if ending:
                out[b, :, a] = part[n]
            else:
                out[b, a] = part[n]
    return out
