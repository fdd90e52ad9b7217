"""bf16 tensor-core path against the CPU oracle.

Bar (per workload): max |gpu - oracle| <= 2e-2 and ||gpu - oracle||_F /
||oracle||_F <= 5e-3. The oracle runs in float64 on exactly the bf16 values the
kernels consume. Every workload, the full-size ones included, is compared
element by element on every cell, in the same launch configuration the
benchmark uses (the oracle's lines spread over spawned processes).
"""
import math

import numpy as np
import pytest
import torch

import oracle.tri_attn_oracle as O
from pair_representation_triangular_gb300 import binding as tb
from pair_representation_triangular_gb300 import workloads as W
from tests import helpers as H
from tests import oracle_pool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from pair_representation_triangular_gb300 import build
    build.build()
    tb.load_library()


@pytest.mark.parametrize("name", W.WORKLOAD_ORDER[2:])
@pytest.mark.parametrize("mode", [0, 1])
def test_bf16_workloads(name, mode):
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w)
    got = H.run_forward(w, inp, mode)[0]
    assert np.all(np.isfinite(got))
    ref = oracle_pool.oracle_forward(w, mode)
    H.assert_parity(w, got, ref)


SMALL = [1, 2, 3, 17, 33, 64, 65, 127, 129, 200]


@pytest.mark.parametrize("N", SMALL)
@pytest.mark.parametrize("mode", [0, 1])
def test_bf16_small_shapes(N, mode):
    w = W.custom(1 + (N % 2), N, 128, 4, "bf16", "bernoulli", seed=2000 + N)
    inp = W.make_inputs(w)
    got = H.run_forward(w, inp, mode)[0]
    ref = O.forward(inp["x"], inp["pair_mask"], inp["params"], w.h, mode)
    H.assert_parity(w, got, ref)


@pytest.mark.parametrize("mode", [0, 1])
def test_bf16_fully_masked_rows_and_queries(mode):
    w = W.custom(1, 150, 128, 4, "bf16", "padded", n_valid=130, seed=31)
    inp = W.make_inputs(w)
    inp["pair_mask"][0, 7, :] = 0              # a fully masked row inside the valid block
    inp["pair_mask"][0, 9, :] = 0
    inp["pair_mask"][0, 9, 64] = 1             # a row that keeps one key only
    got = H.run_forward(w, inp, mode)[0]
    ref = O.forward(inp["x"], inp["pair_mask"], inp["params"], w.h, mode)
    H.assert_parity(w, got, ref)


def test_bf16_rerun_is_bit_identical():
    w = W.custom(1, 96, 128, 4, "bf16", "bernoulli", seed=41)
    inp = W.make_inputs(w)
    a, b = H.run_forward(w, inp, 0, repeats=2)
    assert np.array_equal(a, b)


def test_bf16_forward_host_matches_device():
    w = W.custom(1, 80, 128, 4, "bf16", "bernoulli", seed=42)
    inp = W.make_inputs(w)
    mod = tb.TriangularAttention(w.B, w.N, w.D, w.h, tb.TRI_ATTN_BF16, 0, H.device_params(inp, w))
    try:
        xh = torch.from_numpy(inp["x"]).to(torch.bfloat16).pin_memory()
        mh = torch.from_numpy(inp["pair_mask"]).pin_memory()
        oh = torch.empty_like(xh).pin_memory()
        mod.forward_host(xh, mh, oh)
        od = mod.forward(xh.cuda(), mh.cuda())
        assert mod.sync_check() == tb.TRI_ATTN_OK
        assert torch.equal(oh, od.cpu())
    finally:
        mod.close()


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_bf16_logits_rising_past_the_reference_max(mode):
    """Large pair biases rising along the keys: those of keys 64..127 sit
    56..80 log2 units above the first tile's and those of keys >= 128 at ~115
    (mode 2: the ending node, where the same construction on the grid's rows
    feeds the bias of the column lines). The bias plane holds each (head,
    query) row minus its largest entry and the exponentials use the fixed
    reference 0, so the weights come out right without any rescaling. x and Wb
    are bf16-exact: channel 0 carries a spike of 8 (keys 64..127) or 64 (keys
    >= 128), and Wb reads channel 0 alone (8.0 per head)."""
    w = W.custom(1, 200, 128, 4, "bf16", "bernoulli", seed=61)
    inp = W.make_inputs(w)
    x = inp["x"]
    if mode & tb.TRI_ATTN_ENDING_NODE:
        x[0, 64:128, :, 0] = 8.0
        x[0, 128:, :, 0] = 64.0
    else:
        x[0, :, 64:128, 0] = 8.0
        x[0, :, 128:, 0] = 64.0
    Wb = np.zeros_like(inp["params"]["Wb"])
    Wb[:, 0] = 8.0
    inp["params"]["Wb"] = Wb
    got = H.run_forward(w, inp, mode)[0]
    if mode & tb.TRI_ATTN_ENDING_NODE:
        ref = O.forward_ending(inp["x"], inp["pair_mask"], inp["params"], w.h, mode & 1)
    else:
        ref = O.forward(inp["x"], inp["pair_mask"], inp["params"], w.h, mode)
    H.assert_parity(w, got, ref)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_bf16_logits_far_below_zero(mode):
    """Every pair bias about -141 log2 units, nearly the same for every key of
    a row: the plane subtracts each row's largest entry, so the weights follow
    S alone without any underflow. Channel 0 of every cell carries -64
    (bf16-exact) and Wb reads channel 0 alone (8.0 per head)."""
    w = W.custom(1, 150, 128, 4, "bf16", "bernoulli", seed=62)
    inp = W.make_inputs(w)
    inp["x"][..., 0] = -64.0
    Wb = np.zeros_like(inp["params"]["Wb"])
    Wb[:, 0] = 8.0
    inp["params"]["Wb"] = Wb
    got = H.run_forward(w, inp, mode)[0]
    if mode & tb.TRI_ATTN_ENDING_NODE:
        ref = O.forward_ending(inp["x"], inp["pair_mask"], inp["params"], w.h, mode & 1)
    else:
        ref = O.forward(inp["x"], inp["pair_mask"], inp["params"], w.h, mode)
    H.assert_parity(w, got, ref)


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_bf16_pair_bias_spread_wide(mode):
    """Pair biases of about +-30..60 (natural units), distinct per cell and
    sign: the bias plane is fp16, stored per (head, query) row minus the row's
    largest entry so that the entries carrying the weight are small and
    precise (an fp16 plane of the raw log2(e)-scaled values misses the bar by
    about 2x at these sizes). Channel 0 of each cell carries a bf16-exact value
    of magnitude in [2, 3.75] and random sign, which LayerNorm leaves close to
    itself, and Wb reads channel 0 alone with weight 16."""
    w = W.custom(1, 160, 128, 4, "bf16", "bernoulli", seed=63)
    inp = W.make_inputs(w)
    rng = np.random.default_rng(64)
    mag = np.round(rng.uniform(2.0, 3.75, size=w.cells) * 64.0) / 64.0
    sign = rng.choice([-1.0, 1.0], size=w.cells)
    inp["x"][..., 0] = (mag * sign).reshape(w.B, w.N, w.N).astype(inp["x"].dtype)
    Wb = np.zeros_like(inp["params"]["Wb"])
    Wb[:, 0] = 16.0
    inp["params"]["Wb"] = Wb
    got = H.run_forward(w, inp, mode)[0]
    if mode & tb.TRI_ATTN_ENDING_NODE:
        ref = O.forward_ending(inp["x"], inp["pair_mask"], inp["params"], w.h, mode & 1)
    else:
        ref = O.forward(inp["x"], inp["pair_mask"], inp["params"], w.h, mode)
    H.assert_parity(w, got, ref)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_bf16_exact_rows_for_logits_beyond_range(mode):
    """One key of every line carries S = q.k/sqrt(d) of about +180 log2 units
    for head 0 (q reads channel 0 = 2 of every cell, k reads channel 1, which
    is 0 except a spike of 64 at one key position): P = 2^x overflows, the row
    sum leaves [2^-16, 2^100) and the unit epilogue recomputes those rows
    exactly (its own max, fp32). The weights are then one-hot on that key, so
    bf16 rounding of q and k does not matter. Other heads have q = k = 0."""
    w = W.custom(1, 130, 128, 4, "bf16", "bernoulli", seed=66)
    inp = W.make_inputs(w)
    x = inp["x"]
    x[..., 0] = 2.0
    x[..., 1] = 0.0
    spike = 37                                   # key position carrying the spike
    if mode & tb.TRI_ATTN_ENDING_NODE:
        x[0, spike, :, 1] = 64.0                 # keys of column lines are grid rows
    else:
        x[0, :, spike, 1] = 64.0
    P = inp["params"]
    d = w.D // w.h
    P["Wq"] = np.zeros_like(P["Wq"])
    P["Wk"] = np.zeros_like(P["Wk"])
    P["Wq"][:d, 0] = 1.0
    P["Wk"][:d, 1] = 1.0
    got = H.run_forward(w, inp, mode)[0]
    if mode & tb.TRI_ATTN_ENDING_NODE:
        ref = O.forward_ending(inp["x"], inp["pair_mask"], inp["params"], w.h, mode & 1)
    else:
        ref = O.forward(inp["x"], inp["pair_mask"], inp["params"], w.h, mode)
    H.assert_parity(w, got, ref)


@pytest.mark.parametrize("mode", [0, 2])
def test_bf16_kept_keys_far_below_a_dropped_maximum(mode):
    """Row-key reading, padded mask (the first 100 of 130 residues kept): keys
    >= 100 of every query carry a pair bias of about +88 (natural units) and
    the kept keys about -88. The bias plane's row maximum sits at a dropped
    key, so every kept key lies about 250 log2 units below it: P underflows,
    the row sums fall below 2^-16 and the unit epilogue recomputes those rows
    exactly from the fp32 bias (the fp16 plane would be too coarse there).
    Channel 2 carries +-40 (bf16-exact) and Wb reads it alone (8.0 per head)."""
    w = W.custom(1, 130, 128, 4, "bf16", "padded", n_valid=100, seed=67)
    inp = W.make_inputs(w)
    x = inp["x"]
    if mode & tb.TRI_ATTN_ENDING_NODE:           # key k of column j is cell (k, j)
        x[0, :100, :, 2] = -40.0
        x[0, 100:, :, 2] = 40.0
    else:                                        # key k of row i is cell (j, k) for query j
        x[0, :, :100, 2] = -40.0
        x[0, :, 100:, 2] = 40.0
    Wb = np.zeros_like(inp["params"]["Wb"])
    Wb[:, 2] = 8.0
    inp["params"]["Wb"] = Wb
    got = H.run_forward(w, inp, mode)[0]
    if mode & tb.TRI_ATTN_ENDING_NODE:
        ref = O.forward_ending(inp["x"], inp["pair_mask"], inp["params"], w.h, mode & 1)
    else:
        ref = O.forward(inp["x"], inp["pair_mask"], inp["params"], w.h, mode)
    H.assert_parity(w, got, ref)


def test_bf16_large_grid_sampled_rows():
    """N = 2048 with 2000 residues kept: 32 key tiles per unit and 43 712 work
    units over the 152-CTA grid; whole rows at the edges, tile and row-group
    boundaries and the padding are compared with the oracle."""
    w = W.custom(1, 2048, 128, 4, "bf16", "padded", n_valid=2000, seed=81)
    inp = W.make_inputs(w)
    got = H.run_forward(w, inp, 0)[0]
    rows = sorted({(0, i) for i in (0, 1, 63, 64, 127, 128, 1023, 1024, 1999, 2000, 2046, 2047)})
    ref = O.forward_rows(inp["x"], inp["pair_mask"], inp["params"], w.h, rows, 0)
    H.assert_parity(w, np.stack([got[b, i] for b, i in rows]), ref)
    assert np.all(np.isfinite(got))


@pytest.mark.parametrize("B,N,mode", [(2, 129, 1), (1, 129, 0), (1, 129, 2), (2, 129, 2),
                                      (2, 129, 3), (1, 300, 2)])
def test_bf16_forward_host_pipelined_matches_device(B, N, mode):
    """The host-buffer entry point moves x in four chunks overlapped with the
    first kernel, then runs the attention kernel in chunks of whole waves of
    its work units (three to eight here, one spanning both batch entries when
    B = 2; a chunk finishes the lines of the row groups it completes) and
    copies each chunk's finished lines back while the next runs: grid rows in
    cell order for the starting node; for the ending node grid columns, formed
    by the output kernel in column-ordered tiles (ragged at the column's end:
    129 or 300 rows) and copied back with one strided copy per batch entry. In
    query-key mode the first kernel also reads the mask, which must have
    landed. The result must equal the device-buffer forward bit for bit."""
    w = W.custom(B, N, 128, 4, "bf16", "bernoulli", seed=43)
    inp = W.make_inputs(w)
    mod = tb.TriangularAttention(w.B, w.N, w.D, w.h, tb.TRI_ATTN_BF16, mode, H.device_params(inp, w))
    try:
        xh = torch.from_numpy(inp["x"]).to(torch.bfloat16).pin_memory()
        mh = torch.from_numpy(inp["pair_mask"]).pin_memory()
        oh = torch.full_like(xh, float("nan")).pin_memory()
        mod.forward_host(xh, mh, oh)
        od = mod.forward(xh.cuda(), mh.cuda())
        assert mod.sync_check() == tb.TRI_ATTN_OK
        assert torch.equal(oh, od.cpu())
    finally:
        mod.close()


@pytest.mark.parametrize("mode", [0, 2])
def test_bf16_forward_host_full_size_matches_device(mode):
    """The host-buffer forward at the benchmark workload (B=1, N=768, 700 of 768
    residues kept): x in eight chunks, the attention kernel in seven equal
    chunks of whole waves and the output copied back chunk by chunk, as the
    benchmark's end-to-end figure times it; bit-equal to the device-buffer
    forward (starting and ending node)."""
    w = W.WORKLOADS["b1-n768-d128-h4-bf16-pad700"]
    inp = W.make_inputs(w)
    mod = tb.TriangularAttention(w.B, w.N, w.D, w.h, tb.TRI_ATTN_BF16, mode, H.device_params(inp, w))
    try:
        xh = torch.from_numpy(inp["x"]).to(torch.bfloat16).pin_memory()
        mh = torch.from_numpy(inp["pair_mask"]).pin_memory()
        oh = torch.full_like(xh, float("nan")).pin_memory()
        mod.forward_host(xh, mh, oh)
        od = mod.forward(xh.cuda(), mh.cuda())
        assert mod.sync_check() == tb.TRI_ATTN_OK
        assert torch.equal(oh, od.cpu())
    finally:
        mod.close()


@pytest.mark.parametrize("mode", [0, 1])
def test_bf16_large_common_offset(mode):
    """Cells whose channels share a large offset (x = 40 + N(0, 1), rounded to
    bf16: mean 40, standard deviation 1). The projection kernel takes the
    LayerNorm statistics in one pass shifted by each cell's first channel and
    folds gamma and beta into the pair-bias weights; an unshifted sum of
    squares would lose the variance to cancellation here."""
    w = W.custom(1, 130, 128, 4, "bf16", "bernoulli", seed=65)
    inp = W.make_inputs(w)
    inp["x"] = (inp["x"].astype(np.float64) + 40.0).astype(np.float32)
    inp["x"] = torch.from_numpy(inp["x"]).to(torch.bfloat16).float().numpy()
    got = H.run_forward(w, inp, mode)[0]
    ref = O.forward(inp["x"], inp["pair_mask"], inp["params"], w.h, mode)
    H.assert_parity(w, got, ref)


@pytest.mark.parametrize("mode", [0, 1])
def test_bf16_value_weights_scaled_into_fp16_range(mode):
    """Wv times 2^12 and Wo times 2^-12 (both exact in bf16): the output is that
    of ordinary weights, but the bound on |v| over all inputs exceeds the fp16
    range, so the library stores v times a power of 2 below 1 (carried by the
    resident Wv rows) and divides it out of the attention output."""
    w = W.custom(1, 130, 128, 4, "bf16", "bernoulli", seed=66)
    inp = W.make_inputs(w)
    inp["params"]["Wv"] = (inp["params"]["Wv"].astype(np.float64) * 4096.0).astype(np.float32)
    inp["params"]["Wo"] = (inp["params"]["Wo"].astype(np.float64) / 4096.0).astype(np.float32)
    mod = tb.TriangularAttention(w.B, w.N, w.D, w.h, tb.TRI_ATTN_BF16, mode, H.device_params(inp, w))
    try:
        x = torch.from_numpy(inp["x"]).to("cuda", torch.bfloat16)
        m = torch.from_numpy(inp["pair_mask"]).cuda()
        got = mod.forward(x, m).double().cpu().numpy()
        assert mod.sync_check() == tb.TRI_ATTN_OK
        v_got = mod.intermediate("v").double().cpu().numpy().reshape(-1, w.D)
    finally:
        mod.close()
    P = {k: v.astype(np.float64) for k, v in inp["params"].items()}
    x_hat = O.layer_norm(inp["x"].astype(np.float64), P["gamma"], P["beta"])
    v_ref = O.project(x_hat, P)[2].reshape(-1, w.D)
    scale = float(np.sum(v_got * v_ref) / np.sum(v_ref * v_ref))
    k = round(-math.log2(scale))
    assert k >= 1 and abs(scale * 2.0 ** k - 1.0) < 1e-3, scale
    assert np.all(np.isfinite(v_got)) and np.abs(v_got).max() < 32768.0
    H.assert_parity(w, got, O.forward(inp["x"], inp["pair_mask"], inp["params"], w.h, mode))


@pytest.mark.parametrize("D,h", [(128, 4), (64, 1)])
@pytest.mark.parametrize("mode", [0, 2, 1])
def test_bf16_trailing_dropped_key_tiles(D, h, mode):
    """Row-key reading: the attention skips the trailing 64-key sub-tiles that
    every line of a work unit drops. Lines keep keys 0 .. e - 1 with e cycling
    through tile edges and their neighbours, a line that keeps no key (weight
    on every real key), and lines with holes, so that units mix lines needing
    1 to 4 sub-tiles of N = 200 (and 1 to 2 of N = 100); the ending node reads
    the same pattern along columns. The query-key reading (mode 1) takes every
    sub-tile and is checked on the same mask."""
    for B, N in ((2, 200), (1, 100)):
        w = W.custom(B, N, D, h, "bf16", "bernoulli", seed=9700 + N + D + mode)
        inp = W.make_inputs(w)
        ext = [0, 1, 63, 64, 65, 127, 128, 129, 150, N, 7, 64]
        keep = np.zeros((B, N, N), np.int32)
        for b in range(B):
            for i in range(N):
                e = min(ext[(i + 5 * b) % len(ext)], N)
                keep[b, i, :e] = 1
                if i % 7 == 3 and e > 10:
                    keep[b, i, 2:e:3] = 0           # holes inside the kept range
        inp["pair_mask"] = keep.transpose(0, 2, 1).copy() if mode & tb.TRI_ATTN_ENDING_NODE else keep
        got = H.run_forward(w, inp, mode)[0]
        H.assert_parity(w, got, _oracle(inp, w, mode))


# Every (D, h) the tensor-core kernels are built for: D in {32, 64, 128} and
# d = D / h in {16, 32, 64} (R = 3 lines per attention unit for d = 16, 32;
# R = 2 and 64-key K/V stages for d = 64).
TC_SHAPES = [(32, 2), (32, 1), (64, 4), (64, 2), (64, 1), (128, 8), (128, 4), (128, 2)]


def _oracle(inp, w, mode):
    if mode & tb.TRI_ATTN_ENDING_NODE:
        return O.forward_ending(inp["x"], inp["pair_mask"], inp["params"], w.h, mode & 1)
    return O.forward(inp["x"], inp["pair_mask"], inp["params"], w.h, mode)


@pytest.mark.parametrize("D,h", TC_SHAPES)
@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_bf16_every_tensor_core_shape(D, h, mode):
    """Each shape of the tensor-core kernels, both mask readings, both nodes, at
    N = 130: two 128-query tiles, three 64-key sub-tiles, 133 cell tiles, each
    with a ragged tail."""
    B = 2 if D == 32 else 1
    w = W.custom(B, 130, D, h, "bf16", "bernoulli", seed=9100 + D + h)
    inp = W.make_inputs(w)
    mod = tb.TriangularAttention(B, w.N, D, h, tb.TRI_ATTN_BF16, mode, H.device_params(inp, w))
    try:
        assert tb.tri_attn_kernel_path(mod.handle) == tb.TRI_ATTN_PATH_TENSOR_CORE
    finally:
        mod.close()
    got = H.run_forward(w, inp, mode)[0]
    H.assert_parity(w, got, _oracle(inp, w, mode))


@pytest.mark.parametrize("D,h", [(64, 4), (64, 1), (32, 2)])
@pytest.mark.parametrize("N", [1, 3, 65, 129, 200])
def test_bf16_tensor_core_shapes_ragged(D, h, N):
    """The head dimensions 16 and 64 and the smallest pair dimension at sizes
    from a single cell to several tiles plus a tail (starting node with the
    query-key reading on odd N, the ending node with the row-key reading on
    even N)."""
    mode = 1 if N % 2 else 2
    w = W.custom(1 + (N % 2), N, D, h, "bf16", "bernoulli", seed=9300 + N + D + h)
    inp = W.make_inputs(w)
    got = H.run_forward(w, inp, mode)[0]
    H.assert_parity(w, got, _oracle(inp, w, mode))


def test_bf16_benchmark_shape_takes_the_tensor_core_path():
    w = W.custom(1, 8, 128, 4, "bf16", "ones", seed=1)
    inp = W.make_inputs(w)
    mod = tb.TriangularAttention(1, 8, 128, 4, tb.TRI_ATTN_BF16, 0, H.device_params(inp, w))
    try:
        assert tb.tri_attn_kernel_path(mod.handle) == tb.TRI_ATTN_PATH_TENSOR_CORE
    finally:
        mod.close()
