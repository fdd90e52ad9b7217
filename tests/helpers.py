"""Shared test plumbing: inputs to device tensors, handles, error metrics."""
import numpy as np
import torch

from pair_representation_triangular_gb300 import binding as tb

TOL_F32_MAX_ABS = 1e-4          # fp32 path: max |gpu - oracle|
TOL_BF16_MAX_ABS = 2e-2         # bf16 path: max |gpu - oracle| ...
TOL_BF16_REL_FRO = 5e-3         # ... and ||gpu - oracle||_F / ||oracle||_F


def dtype_code(w):
    return tb.TRI_ATTN_F32 if w.dtype == "f32" else tb.TRI_ATTN_BF16


def torch_dtype(w):
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def device_params(inp, w, device="cuda"):
    td = torch_dtype(w)
    return {k: torch.from_numpy(np.ascontiguousarray(v)).to(device=device, dtype=td)
            for k, v in inp["params"].items()}


def run_forward(w, inp, mask_mode=0, repeats=1):
    """Create a handle, run the forward pass `repeats` times; returns the list of
    float64 numpy outputs and the final sync status."""
    td = torch_dtype(w)
    x = torch.from_numpy(inp["x"]).to("cuda", dtype=td)
    m = torch.from_numpy(inp["pair_mask"]).to("cuda")
    mod = tb.TriangularAttention(w.B, w.N, w.D, w.h, dtype_code(w), mask_mode,
                                 device_params(inp, w))
    outs = []
    try:
        for _ in range(repeats):
            out = mod.forward(x, m)
            status = mod.sync_check()
            assert status == tb.TRI_ATTN_OK, tb.tri_attn_status_string(status)
            outs.append(out.to(torch.float64).cpu().numpy())
    finally:
        mod.close()
    return outs


def errors(got, ref):
    diff = got - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    rel_fro = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))
    return max_abs, rel_fro


def assert_parity(w, got, ref):
    assert np.all(np.isfinite(got)), "non-finite output"
    max_abs, rel_fro = errors(got, ref)
    if w.dtype == "f32":
        assert max_abs <= TOL_F32_MAX_ABS, f"{w.name}: max abs err {max_abs:.3e}"
    else:
        assert max_abs <= TOL_BF16_MAX_ABS and rel_fro <= TOL_BF16_REL_FRO, \
            f"{w.name}: max abs err {max_abs:.3e}, rel Frobenius {rel_fro:.3e}"
    return max_abs, rel_fro
