"""Seeded synthetic workloads for triangular self-attention (both node variants).

This module only draws inputs. It holds none of the method's arithmetic, so both
the CUDA path and the CPU oracle can take their inputs from it without sharing
any computation.

Shapes follow the benchmark module on the POPCORNBENCH pages (triangular
self-attention, "Kimi-K2.6 l2_p6": module constants and ``get_inputs``), widened
to the five benchmark configurations listed in ``WORKLOADS``.

Recipe, drawn in this fixed order from ``numpy.random.default_rng(seed)``:

1. ``x`` ~ N(0, 1) of shape (B, N, N, D). With ``cell_scale`` every cell
   (b, r, c) is multiplied by one U(0.5, 2) draw.
2. ``pair_mask`` (int32, (B, N, N), nonzero = keep):
   * ``bernoulli``: Bernoulli(0.9); a row r of ``pair_mask[b]`` that came out
     all zero gets ``pair_mask[b, r, r] = 1``, so every row keeps a key;
   * ``ones``: all ones;
   * ``padded``: ``s[r] * s[c]`` with ``s`` one on the first ``n_valid``
     residues and zero after.
3. LayerNorm ``gamma = 1 + 0.1 N(0,1)``, ``beta = 0.1 N(0,1)``.
4. ``Wq, Wk, Wv, Wg, bg, Wb, Wo, bo`` ~ U(-1/sqrt(D), 1/sqrt(D)) in that
   order (fan_in = D for every Linear); ``Wb`` is (h, D), the rest (D, D)/(D,).
5. For bf16 workloads, ``x`` and every parameter are rounded to bf16
   (round-to-nearest-even). Arrays are returned as float32 holding exactly the
   values the kernels consume.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

PARAM_NAMES = ("gamma", "beta", "Wq", "Wk", "Wv", "Wg", "bg", "Wb", "Wo", "bo")


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    N: int
    D: int
    h: int
    dtype: str          # "f32" or "bf16"
    mask: str           # "bernoulli" | "ones" | "padded"
    n_valid: int = 0    # residues kept by a "padded" mask
    cell_scale: bool = False
    seed: int = 0

    @property
    def d(self) -> int:
        return self.D // self.h

    @property
    def cells(self) -> int:
        return self.B * self.N * self.N


WORKLOADS = {
    w.name: w
    for w in (
        Workload("b2-n32-d64-h4-f32", 2, 32, 64, 4, "f32", "bernoulli", seed=0),
        Workload("b1-n128-d128-h4-f32", 1, 128, 128, 4, "f32", "bernoulli", seed=1),
        Workload("b1-n256-d128-h4-bf16", 1, 256, 128, 4, "bf16", "ones", seed=2),
        Workload("b1-n384-d128-h4-bf16-pad320", 1, 384, 128, 4, "bf16", "padded",
                 n_valid=320, seed=3),
        Workload("b1-n768-d128-h4-bf16-pad700", 1, 768, 128, 4, "bf16", "padded",
                 n_valid=700, cell_scale=True, seed=4),
    )
}
WORKLOAD_ORDER = list(WORKLOADS)


def custom(B, N, D, h, dtype="f32", mask="bernoulli", n_valid=0, cell_scale=False,
           seed=0) -> Workload:
    """A workload of any shape, drawn with the same recipe."""
    return Workload(f"b{B}-n{N}-d{D}-h{h}-{dtype}-{mask}", B, N, D, h, dtype, mask,
                    n_valid, cell_scale, seed)


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even), kept as float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32)
    # NaN/inf never occur in these draws; keep them unchanged if they ever do.
    bad = ~np.isfinite(a)
    if bad.any():
        out = out.copy()
        out[bad] = a[bad]
    return out


def make_mask(rng: np.random.Generator, w: Workload) -> np.ndarray:
    B, N = w.B, w.N
    if w.mask == "bernoulli":
        m = (rng.random((B, N, N)) < 0.9).astype(np.int32)
        for b in range(B):
            empty = np.flatnonzero(m[b].sum(axis=1) == 0)
            m[b, empty, empty] = 1
        return m
    if w.mask == "ones":
        return np.ones((B, N, N), np.int32)
    if w.mask == "padded":
        s = (np.arange(N) < w.n_valid).astype(np.int32)
        return np.broadcast_to(np.outer(s, s), (B, N, N)).astype(np.int32).copy()
    raise ValueError(f"unknown mask kind {w.mask!r}")


def make_inputs(w: Workload) -> dict:
    """Draw (x, pair_mask, params) for workload ``w``; see the module docstring."""
    rng = np.random.default_rng(w.seed)
    B, N, D, h = w.B, w.N, w.D, w.h
    if D % h:
        raise ValueError("D must be a multiple of h")
    x = rng.standard_normal((B, N, N, D), dtype=np.float32)
    if w.cell_scale:
        x *= rng.uniform(0.5, 2.0, size=(B, N, N, 1)).astype(np.float32)
    mask = make_mask(rng, w)
    bound = 1.0 / np.sqrt(D)
    p = {
        "gamma": (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32),
        "beta": (0.1 * rng.standard_normal(D)).astype(np.float32),
    }
    for name, shape in (("Wq", (D, D)), ("Wk", (D, D)), ("Wv", (D, D)), ("Wg", (D, D)),
                        ("bg", (D,)), ("Wb", (h, D)), ("Wo", (D, D)), ("bo", (D,))):
        p[name] = rng.uniform(-bound, bound, size=shape).astype(np.float32)
    if w.dtype == "bf16":
        x = round_to_bf16(x)
        p = {k: round_to_bf16(v) for k, v in p.items()}
    elif w.dtype != "f32":
        raise ValueError(f"unknown dtype {w.dtype!r}")
    return {"x": x, "pair_mask": mask, "params": p}


def with_seed(w: Workload, seed: int) -> Workload:
    return replace(w, seed=seed)
