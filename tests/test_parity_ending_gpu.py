"""Ending-node variant (mode flag TRI_ATTN_ENDING_NODE) against the oracle's
column-wise statement of it, on both paths and both mask readings.

Same bars as the starting node: fp32 max |gpu - oracle| <= 1e-4; bf16 max abs
<= 2e-2 and relative Frobenius <= 5e-3. Full-size bf16 workloads are compared
on whole columns (b, :, j) — edges, tile and row-group boundaries and the first
padded columns — in the launch configuration the benchmark uses.
"""
import numpy as np
import pytest

import oracle.tri_attn_oracle as O
from pair_representation_triangular_gb300 import binding as tb
from pair_representation_triangular_gb300 import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu

END = tb.TRI_ATTN_ENDING_NODE


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from pair_representation_triangular_gb300 import build
    build.build()
    tb.load_library()


def _cols_for(w):
    N = w.N
    cols = {0, 1, 3, 4, 5, 63, 64, 127, 128, 129, N // 2, N - 2, N - 1}
    if w.mask == "padded":
        cols |= {w.n_valid - 1, w.n_valid, w.n_valid + 1}
    return sorted((b, j) for b in range(w.B) for j in cols if 0 <= j < N)


@pytest.mark.parametrize("name", W.WORKLOAD_ORDER)
@pytest.mark.parametrize("mode", [0, 1])
def test_ending_workloads(name, mode):
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w)
    got = H.run_forward(w, inp, mode | END)[0]
    if w.N <= 256:
        ref = O.forward_ending(inp["x"], inp["pair_mask"], inp["params"], w.h, mode)
        H.assert_parity(w, got, ref)
    else:
        cols = _cols_for(w)
        ref = O.forward_ending_columns(inp["x"], inp["pair_mask"], inp["params"], w.h, cols, mode)
        sub = np.stack([got[b, :, j] for b, j in cols])
        H.assert_parity(w, sub, ref)
    assert np.all(np.isfinite(got))


@pytest.mark.parametrize("N", [1, 2, 3, 33, 65, 129, 200])
@pytest.mark.parametrize("mode", [0, 1])
def test_ending_bf16_small_shapes(N, mode):
    w = W.custom(1 + (N % 2), N, 128, 4, "bf16", "bernoulli", seed=5000 + N)
    inp = W.make_inputs(w)
    got = H.run_forward(w, inp, mode | END)[0]
    ref = O.forward_ending(inp["x"], inp["pair_mask"], inp["params"], w.h, mode)
    H.assert_parity(w, got, ref)


@pytest.mark.parametrize("B,N,D,h", [(1, 1, 32, 1), (2, 17, 32, 4), (1, 33, 64, 2),
                                     (1, 129, 64, 4), (1, 20, 128, 4), (1, 70, 128, 1)])
@pytest.mark.parametrize("mode", [0, 1])
def test_ending_f32_small_shapes(B, N, D, h, mode):
    w = W.custom(B, N, D, h, "f32", "bernoulli", seed=6000 + N + D + h)
    inp = W.make_inputs(w)
    got = H.run_forward(w, inp, mode | END)[0]
    ref = O.forward_ending(inp["x"], inp["pair_mask"], inp["params"], h, mode)
    H.assert_parity(w, got, ref)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", [0, 1])
def test_ending_fully_masked_columns(dtype, mode):
    w = W.custom(1, 150, 128, 4, dtype, "padded", n_valid=130, seed=51)
    inp = W.make_inputs(w)
    inp["pair_mask"][0, :, 7] = 0              # a fully masked column inside the valid block
    inp["pair_mask"][0, :, 9] = 0
    inp["pair_mask"][0, 64, 9] = 1             # a column that keeps one key only
    got = H.run_forward(w, inp, mode | END)[0]
    ref = O.forward_ending(inp["x"], inp["pair_mask"], inp["params"], w.h, mode)
    H.assert_parity(w, got, ref)


def test_ending_differs_from_starting():
    """The flag changes the result (the two variants agree only on symmetric
    inputs), so a path that ignored it could not pass the tests above by luck."""
    w = W.custom(1, 40, 128, 4, "bf16", "bernoulli", seed=52)
    inp = W.make_inputs(w)
    start = H.run_forward(w, inp, 0)[0]
    end = H.run_forward(w, inp, END)[0]
    assert float(np.max(np.abs(start - end))) > 10 * H.TOL_BF16_MAX_ABS


def _sweep_cases():
    rng = np.random.default_rng(2026)
    cases = []
    for _ in range(12):
        B = int(rng.integers(1, 4))
        N = int(rng.integers(1, 260))
        mode = int(rng.integers(0, 4))                 # mask reading | ending-node flag
        cases.append((B, N, mode))
    return cases


@pytest.mark.parametrize("B,N,mode", _sweep_cases())
def test_bf16_seeded_shape_sweep(B, N, mode):
    """Seeded random shapes (B 1-3, N 1-259, both nodes, both mask readings)
    on the tensor-core path against the oracle."""
    w = W.custom(B, N, 128, 4, "bf16", "bernoulli", seed=7000 + 31 * N + B)
    inp = W.make_inputs(w)
    got = H.run_forward(w, inp, mode)[0]
    if mode & END:
        ref = O.forward_ending(inp["x"], inp["pair_mask"], inp["params"], w.h, mode & 1)
    else:
        ref = O.forward(inp["x"], inp["pair_mask"], inp["params"], w.h, mode)
    H.assert_parity(w, got, ref)
