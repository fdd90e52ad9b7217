"""Kernel-by-kernel parity: each kernel's output against the oracle's step run on
that kernel's own GPU inputs, so an error is attributed to one kernel.

  K1  q, k, v, g and the bias plane   vs  oracle layer_norm + project  (on x)
  K2  o                               vs  oracle row_attention (on GPU q, k, v, bias)
  K3  out                             vs  oracle output_projection (on GPU g, o)
"""
import math

import numpy as np
import pytest
import torch

import oracle.tri_attn_oracle as O
from pair_representation_triangular_gb300 import binding as tb
from pair_representation_triangular_gb300 import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu

LOG2E = 1.0 / math.log(2.0)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from pair_representation_triangular_gb300 import build
    build.build()
    tb.load_library()


def _rel_fro(got, ref):
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def _run(w, mode):
    inp = W.make_inputs(w)
    td = H.torch_dtype(w)
    mod = tb.TriangularAttention(w.B, w.N, w.D, w.h, H.dtype_code(w), mode, H.device_params(inp, w))
    x = torch.from_numpy(inp["x"]).to("cuda", td)
    m = torch.from_numpy(inp["pair_mask"]).cuda()
    out = mod.forward(x, m)
    assert mod.sync_check() == tb.TRI_ATTN_OK
    got = {n: mod.intermediate(n).double().cpu().numpy() for n in ("q", "k", "v", "g", "o", "bias")}
    got["out"] = out.double().cpu().numpy()
    mod.close()
    return inp, got


CASES = [(W.custom(1, 130, 128, 4, "bf16", "bernoulli", seed=71), 0),
         (W.custom(1, 130, 128, 4, "bf16", "bernoulli", seed=72), 1),
         (W.custom(2, 33, 64, 4, "f32", "bernoulli", seed=73), 0)]
# The other tensor-core shapes (D, h): each kernel's instantiation on its own.
CASES += [(W.custom(1, 130, D, h, "bf16", "bernoulli", seed=74 + i), i % 2)
          for i, (D, h) in enumerate([(32, 2), (32, 1), (64, 4), (64, 2), (64, 1), (128, 8),
                                      (128, 2)])]


@pytest.mark.parametrize("w,mode", CASES, ids=[f"{w.name}-m{m}" for w, m in CASES])
def test_stage_by_stage(w, mode):
    inp, got = _run(w, mode)
    P = {k: v.astype(np.float64) for k, v in inp["params"].items()}
    bf16 = w.dtype == "bf16"
    tol = 5e-3 if bf16 else 1e-5

    # K1: projections and the bias plane. The tensor-core path stores q times
    # log2(e) / sqrt(d) (the attention's exponentials are powers of 2).
    x_hat = O.layer_norm(inp["x"].astype(np.float64), P["gamma"], P["beta"])
    q, k, v, g, bc = O.project(x_hat, P)
    if bf16:
        got["q"] = got["q"] / (LOG2E / math.sqrt(w.D // w.h))
    for name, ref in (("q", q), ("k", k), ("v", v), ("g", g)):
        assert _rel_fro(got[name], ref) <= tol, name
    bias_ref = O.bias_plane(bc)
    bias_got = got["bias"] / LOG2E if bf16 else got["bias"]
    if bf16:
        # The tensor-core path stores each (head, query) row of the plane minus
        # its largest kept entry (the softmax over keys is unchanged by it).
        dropped = np.zeros(bias_ref.shape, bool)
        if mode == O.MASK_QUERY_KEY:
            dropped = np.broadcast_to((inp["pair_mask"] == 0)[:, None], bias_ref.shape)
            assert np.all(np.isneginf(bias_got[dropped]))
        rowmax = np.where(dropped, -np.inf, bias_ref).max(axis=-1, keepdims=True)
        bias_ref = bias_ref - rowmax
        keep = ~dropped
        assert _rel_fro(bias_got[keep], bias_ref[keep]) <= tol
    else:
        assert _rel_fro(bias_got, bias_ref) <= tol

    # K2: attention on the GPU's own q, k, v and bias
    gb = np.where(np.isneginf(bias_got), 0.0, bias_got)
    B, N, D, h = w.B, w.N, w.D, w.h
    for b in range(B):
        for i in sorted({0, N // 2, N - 1}):
            keep = O.keep_matrix(inp["pair_mask"], b, i, mode)
            o_ref = O.row_attention(got["q"][b, i], got["k"][b, i], got["v"][b, i], gb[b], keep, h)
            assert _rel_fro(got["o"][b, i], o_ref) <= (4e-3 if bf16 else 1e-5), (b, i)

    # K3: gate and output projection on the GPU's own g and o
    out_ref = O.output_projection(got["g"], got["o"], P)
    assert _rel_fro(got["out"], out_ref) <= (3e-3 if bf16 else 1e-5)
