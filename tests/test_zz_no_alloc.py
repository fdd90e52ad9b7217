"""tri_attn_forward_noalloc: the fp32 forward pass for callers that may not
allocate device memory (memory pools or custom allocators that forbid outside
allocations, plugins given only their input and output buffers). It keeps its
intermediates in the library's fixed device scratch instead of a handle's
workspace. Checked through the C ABI against the handle-based tri_attn_forward
and against the CPU oracle on two calls in a row with different inputs, so a
call that read stale scratch from the one before would show; and a problem
beyond the fixed scratch must be refused. This file is collected last on
purpose."""
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


@pytest.mark.parametrize("mode", [0, 1, 2, 3])      # mask reading | ending-node flag
def test_noalloc_matches_forward_on_two_calls(mode):
    for seed in (11, 12):                      # two calls in a row, different inputs
        w = W.custom(2, 32, 64, 4, "f32", "bernoulli", seed=seed)
        inp = W.make_inputs(w)
        params = H.device_params(inp, w)
        x = torch.from_numpy(inp["x"]).cuda()
        m = torch.from_numpy(inp["pair_mask"]).cuda()
        out = torch.full_like(x, float("nan"))
        tb.tri_attn_forward_noalloc(w.B, w.N, w.D, w.h, mode, params, None, x, m, out)
        torch.cuda.synchronize()
        mod = tb.TriangularAttention(w.B, w.N, w.D, w.h, tb.TRI_ATTN_F32, mode, params)
        try:
            ref = mod.forward(x, m)
            assert mod.sync_check() == tb.TRI_ATTN_OK
        finally:
            mod.close()
        got, want = out.double().cpu().numpy(), ref.double().cpu().numpy()
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got - want))) <= H.TOL_F32_MAX_ABS
        if mode & tb.TRI_ATTN_ENDING_NODE:
            oracle = O.forward_ending(inp["x"], inp["pair_mask"], inp["params"], w.h, mode & 1)
        else:
            oracle = O.forward(inp["x"], inp["pair_mask"], inp["params"], w.h, mode)
        H.assert_parity(w, got, oracle)


def test_noalloc_refuses_problems_beyond_its_scratch():
    w = W.custom(1, 128, 128, 4, "f32", "ones", seed=13)   # needs about 42 MB > 16 MiB
    inp = W.make_inputs(w)
    params = H.device_params(inp, w)
    x = torch.from_numpy(inp["x"]).cuda()
    m = torch.from_numpy(inp["pair_mask"]).cuda()
    out = torch.zeros_like(x)
    with pytest.raises(tb.TriAttnError) as e:
        tb.tri_attn_forward_noalloc(w.B, w.N, w.D, w.h, 0, params, None, x, m, out)
    assert e.value.status == tb.TRI_ATTN_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0           # nothing was launched
