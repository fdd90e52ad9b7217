"""Row sharding of one problem over ranks, checked on the CPU with two gloo
ranks (127.0.0.1) running the oracle's steps.

Every quantity of softmax row i (q, k, v, g, o, out of cells (b, i, :)) depends
on row i of the pair representation alone, except the pair bias, which every
row reads at all (j, k). So rank p projects its own rows (LayerNorm, q, k, v, g
and the h bias values of each of its cells), one all-gather assembles the
(B, h, N, N) bias plane, and attention plus the output projection then run on
rank p's rows with no further exchange. The ending node is the same with
columns in place of rows. The gathered output must equal the single-process
oracle. This is the decomposition a multi-GPU build would use (one all-gather
of B*h*N^2 bias values before the attention kernel); the library itself runs
one problem per GPU.
"""
import os
import socket

import numpy as np
import torch
import torch.multiprocessing as mp

import oracle.tri_attn_oracle as O
from pair_representation_triangular_gb300 import workloads as W

B, N, D, H = 2, 6, 16, 4


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    inp = W.make_inputs(W.custom(B, N, D, H, "f32", "bernoulli", seed=71))
    P = {k: v.astype(np.float64) for k, v in inp["params"].items()}
    return inp["x"].astype(np.float64), inp["pair_mask"], P


def _rank_main(rank, world, port, mode, ending, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x, mask, P = _inputs()
        xl = np.swapaxes(x, 1, 2) if ending else x          # lines first: x[b, line, pos]
        per = N // world
        mine = range(rank * per, (rank + 1) * per)
        # local step: LayerNorm and projections of this rank's lines
        x_hat = O.layer_norm(xl[:, mine], P["gamma"], P["beta"])
        q, k, v, g, bias_cells = O.project(x_hat, P)        # bias_cells (B, per, N, h)
        # the one exchange: all-gather of the per-cell bias values
        parts = [torch.empty((B, per, N, H), dtype=torch.float64) for _ in range(world)]
        torch.distributed.all_gather(parts, torch.from_numpy(np.ascontiguousarray(bias_cells)))
        gathered = np.concatenate([p.numpy() for p in parts], axis=1)   # (B, N lines, N, h)
        cells = np.swapaxes(gathered, 1, 2) if ending else gathered      # back to grid (r, c)
        plane = O.bias_plane(cells)
        # local attention and output projection over this rank's lines
        res = np.empty((B, per, N, D))
        for b in range(B):
            for n, a in enumerate(mine):
                if ending:
                    keep, bias_l = O.column_keep(mask, b, a, mode), O.column_bias(plane[b])
                else:
                    keep, bias_l = O.keep_matrix(mask, b, a, mode), plane[b]
                o = O.row_attention(q[b, n], k[b, n], v[b, n], bias_l, keep, H)
                res[b, n] = O.output_projection(g[b, n], o, P)
        outs = [torch.empty((B, per, N, D), dtype=torch.float64) for _ in range(world)]
        torch.distributed.all_gather(outs, torch.from_numpy(res))
        if rank == 0:
            full = np.concatenate([t.numpy() for t in outs], axis=1)
            out["result"] = np.swapaxes(full, 1, 2) if ending else full
    finally:
        torch.distributed.destroy_process_group()


def _run(mode, ending):
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), mode, ending, out), nprocs=world, join=True)
        return out["result"]


def test_row_shards_match_single_process():
    x, mask, P = _inputs()
    for mode in (O.MASK_ROW_KEY, O.MASK_QUERY_KEY):
        np.testing.assert_allclose(_run(mode, False), O.forward(x, mask, P, H, mode),
                                   rtol=0, atol=1e-12)


def test_column_shards_match_single_process_ending_node():
    x, mask, P = _inputs()
    for mode in (O.MASK_ROW_KEY, O.MASK_QUERY_KEY):
        np.testing.assert_allclose(_run(mode, True), O.forward_ending(x, mask, P, H, mode),
                                   rtol=0, atol=1e-12)
