"""Failure detection without a GPU fault: every device-side wait of the
tensor-core kernels is bounded. With the test hook capping waits at one poll,
the first wait that is not already complete gives up; the kernel records a
time-out, drains its own copies and MMAs, frees its tensor memory and returns.
The host sees TRI_ATTN_ERR_DEVICE_TIMEOUT, and the same handle then computes a
correct result once the cap is lifted."""
import numpy as np
import pytest
import torch

import oracle.tri_attn_oracle as O
from pair_representation_triangular_gb300 import binding as tb
from pair_representation_triangular_gb300 import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    from pair_representation_triangular_gb300 import build
    build.build()
    w = W.custom(1, 100, 128, 4, "bf16", "bernoulli", seed=61)
    inp = W.make_inputs(w)
    mod = tb.TriangularAttention(w.B, w.N, w.D, w.h, tb.TRI_ATTN_BF16, 0, H.device_params(inp, w))
    try:
        x = torch.from_numpy(inp["x"]).to("cuda", torch.bfloat16)
        m = torch.from_numpy(inp["pair_mask"]).cuda()
        tb.tri_attn_set_wait_limit(mod.handle, 1)
        mod.forward(x, m)
        assert mod.sync_check() == tb.TRI_ATTN_ERR_DEVICE_TIMEOUT
        assert mod.sync_check() == tb.TRI_ATTN_OK          # the error word was cleared
        tb.tri_attn_set_wait_limit(mod.handle, 0)          # default limit again
        out = mod.forward(x, m)
        assert mod.sync_check() == tb.TRI_ATTN_OK
        ref = O.forward(inp["x"], inp["pair_mask"], inp["params"], w.h, 0)
        H.assert_parity(w, out.double().cpu().numpy(), ref)
    finally:
        mod.close()
