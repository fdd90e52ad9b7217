"""fp32 SIMT path against the CPU oracle, element by element (max abs <= 1e-4)."""
import numpy as np
import pytest
import torch

import oracle.tri_attn_oracle as O
from pair_representation_triangular_gb300 import binding as tb
from pair_representation_triangular_gb300 import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from pair_representation_triangular_gb300 import build
    build.build()
    tb.load_library()


@pytest.mark.parametrize("name", W.WORKLOAD_ORDER[:2])
@pytest.mark.parametrize("mode", [0, 1])
def test_f32_workloads(name, mode):
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w)
    got = H.run_forward(w, inp, mode)[0]
    ref = O.forward(inp["x"], inp["pair_mask"], inp["params"], w.h, mode)
    H.assert_parity(w, got, ref)


SHAPES = [(1, 1, 32, 1), (2, 2, 32, 2), (1, 3, 64, 4), (1, 17, 32, 4), (2, 33, 64, 2),
          (1, 127, 32, 1), (1, 129, 64, 4), (1, 33, 128, 1), (1, 20, 128, 4), (1, 9, 96, 4),
          (1, 130, 256, 2)]   # d = 128: two threads per query, several key chunks


@pytest.mark.parametrize("B,N,D,h", SHAPES)
@pytest.mark.parametrize("mode", [0, 1])
def test_f32_small_shapes(B, N, D, h, mode):
    w = W.custom(B, N, D, h, "f32", "bernoulli", seed=1000 + N + D + h)
    inp = W.make_inputs(w)
    got = H.run_forward(w, inp, mode)[0]
    ref = O.forward(inp["x"], inp["pair_mask"], inp["params"], h, mode)
    H.assert_parity(w, got, ref)


@pytest.mark.parametrize("mode", [0, 1])
def test_f32_fully_masked_rows_and_padding(mode):
    w = W.custom(1, 37, 64, 4, "f32", "padded", n_valid=30, seed=77)
    inp = W.make_inputs(w)
    inp["pair_mask"][0, 3, :] = 0                     # one more fully masked row
    got = H.run_forward(w, inp, mode)[0]
    ref = O.forward(inp["x"], inp["pair_mask"], inp["params"], w.h, mode)
    H.assert_parity(w, got, ref)


def test_f32_rerun_is_bit_identical():
    w = W.WORKLOADS[W.WORKLOAD_ORDER[0]]
    inp = W.make_inputs(w)
    a, b = H.run_forward(w, inp, 0, repeats=2)
    assert np.array_equal(a, b)


def test_f32_forward_host_matches_device():
    w = W.WORKLOADS[W.WORKLOAD_ORDER[0]]
    inp = W.make_inputs(w)
    mod = tb.TriangularAttention(w.B, w.N, w.D, w.h, tb.TRI_ATTN_F32, 0, H.device_params(inp, w))
    try:
        xh = torch.from_numpy(inp["x"]).pin_memory()
        mh = torch.from_numpy(inp["pair_mask"]).pin_memory()
        oh = torch.empty_like(xh).pin_memory()
        mod.forward_host(xh, mh, oh)
        od = mod.forward(xh.cuda(), mh.cuda())
        assert mod.sync_check() == tb.TRI_ATTN_OK
        assert torch.equal(oh, od.cpu())
    finally:
        mod.close()


def test_forward_rejects_overlapping_output():
    w = W.WORKLOADS[W.WORKLOAD_ORDER[0]]
    inp = W.make_inputs(w)
    mod = tb.TriangularAttention(w.B, w.N, w.D, w.h, tb.TRI_ATTN_F32, 0, H.device_params(inp, w))
    try:
        x = torch.from_numpy(inp["x"]).cuda()
        m = torch.from_numpy(inp["pair_mask"]).cuda()
        with pytest.raises(tb.TriAttnError) as e:
            tb.tri_attn_forward(mod.handle, None, x, m, x)
        assert e.value.status == tb.TRI_ATTN_ERR_INVALID_ARG
    finally:
        mod.close()
