"""The seeded input recipe: shapes, mask structure, bf16 rounding, determinism."""
import numpy as np
import torch

from pair_representation_triangular_gb300 import workloads as W


def test_bf16_rounding_matches_torch_cast():
    a = np.random.default_rng(0).standard_normal(100_000).astype(np.float32) * 7
    a[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]     # exact ties: to even
    ref = torch.from_numpy(a).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(W.round_to_bf16(a).view(np.uint32), ref.view(np.uint32))


def test_small_workloads_recipe():
    for name in W.WORKLOAD_ORDER[:3]:
        w = W.WORKLOADS[name]
        inp = W.make_inputs(w)
        assert inp["x"].shape == (w.B, w.N, w.N, w.D)
        assert inp["pair_mask"].dtype == np.int32
        assert (inp["pair_mask"].sum(axis=2) > 0).all()          # a kept key per row
        assert inp["params"]["Wb"].shape == (w.h, w.D)
        again = W.make_inputs(w)
        assert np.array_equal(inp["x"], again["x"])
        if w.dtype == "bf16":
            assert np.array_equal(W.round_to_bf16(inp["x"]), inp["x"])


def test_padded_mask_structure():
    w = W.custom(1, 12, 8, 2, "bf16", "padded", n_valid=9, seed=3)
    m = W.make_inputs(w)["pair_mask"][0]
    s = (np.arange(12) < 9).astype(np.int32)
    assert np.array_equal(m, np.outer(s, s))
