"""Pins for the CPU oracle: closed forms, invariants, special cases that reduce
to library routines, and a hand-derived worked example. Each pin is checked
against the oracle as it stands, and each known-wrong variant of the method
(the mistakes catalogued on the POPCORNBENCH pages, planted here in the oracle
on the CPU) must make at least the named pin fail.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle.tri_attn_oracle as O
from pair_representation_triangular_gb300 import workloads as W
from tests import torch_library_module as TLM

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _inputs(B, N, D, h, seed, mask="bernoulli"):
    inp = W.make_inputs(W.custom(B, N, D, h, "f32", mask, seed=seed))
    P = {k: v.astype(np.float64) for k, v in inp["params"].items()}
    return inp["x"].astype(np.float64), inp["pair_mask"], P


def _t(a):
    return torch.as_tensor(np.asarray(a), dtype=torch.float64)


def _lib_ln(x, P):
    return F.layer_norm(_t(x), (x.shape[-1],), _t(P["gamma"]), _t(P["beta"]), eps=1e-5)


# ----------------------------------------------------------------------------- pins

def pin_n1_closed_form():
    """N = 1: the single softmax weight is 1 whatever the mask, so
    out = Wo (sigmoid(Wg x_hat + bg) * (Wv x_hat)) + bo, built here from
    torch's layer_norm / linear / sigmoid."""
    for mode in (O.MASK_ROW_KEY, O.MASK_QUERY_KEY):
        for mval in (0, 1):
            x, _, P = _inputs(2, 1, 8, 2, seed=11)
            mask = np.full((2, 1, 1), mval, np.int32)
            out = O.forward(x, mask, P, 2, mode)
            xn = _lib_ln(x, P)
            g = torch.sigmoid(F.linear(xn, _t(P["Wg"]), _t(P["bg"])))
            v = F.linear(xn, _t(P["Wv"]))
            ref = F.linear(g * v, _t(P["Wo"]), _t(P["bo"])).numpy()
            np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def pin_rows_sum_to_one():
    """Every softmax row of every head sums to 1; dropped keys weigh exactly 0
    on rows that keep a key."""
    x, mask, P = _inputs(2, 9, 8, 2, seed=12)
    for mode in (O.MASK_ROW_KEY, O.MASK_QUERY_KEY):
        for b, i in ((0, 0), (1, 4), (1, 8)):
            p = O.attention_probs(x, mask, P, 2, b, i, mode)
            np.testing.assert_allclose(p.sum(axis=-1), 1.0, rtol=0, atol=1e-12)
            assert (p >= 0).all()
            keep = O.keep_matrix(mask, b, i, mode)
            assert np.all(p[:, ~keep] == 0.0)


def pin_all_ones_mask_is_no_mask():
    x, _, P = _inputs(1, 7, 8, 2, seed=13)
    ones = np.ones((1, 7, 7), np.int32)
    for mode in (O.MASK_ROW_KEY, O.MASK_QUERY_KEY):
        assert np.array_equal(O.forward(x, ones, P, 2, mode), O.forward(x, None, P, 2, mode))


def pin_relabelling_equivariance():
    """Permuting both grid axes of pair_repr and pair_mask by pi permutes out."""
    x, mask, P = _inputs(2, 8, 8, 4, seed=14)
    pi = np.random.default_rng(5).permutation(8)
    xp = x[:, pi][:, :, pi]
    mp = mask[:, pi][:, :, pi]
    for mode in (O.MASK_ROW_KEY, O.MASK_QUERY_KEY):
        out = O.forward(x, mask, P, 4, mode)
        outp = O.forward(xp, mp, P, 4, mode)
        np.testing.assert_allclose(outp, out[:, pi][:, :, pi], rtol=0, atol=1e-12)


def pin_single_kept_key():
    """A softmax row that keeps exactly one key k* puts weight 1 on it, so
    o = v[b, i, k*] there. Mode row-key: row i keeps k* for every query j.
    Mode query-key: query j keeps k* in every row i."""
    B, N, D, h = 1, 6, 8, 2
    x, _, P = _inputs(B, N, D, h, seed=15)
    xn = _lib_ln(x, P)
    g = torch.sigmoid(F.linear(xn, _t(P["Wg"]), _t(P["bg"])))
    v = F.linear(xn, _t(P["Wv"]))
    i0, k_star = 2, 4
    mask = np.ones((B, N, N), np.int32)
    mask[0, i0, :] = 0
    mask[0, i0, k_star] = 1
    out = O.forward(x, mask, P, h, O.MASK_ROW_KEY)
    ref = F.linear(g[0, i0] * v[0, i0, k_star][None, :], _t(P["Wo"]), _t(P["bo"])).numpy()
    np.testing.assert_allclose(out[0, i0], ref, rtol=0, atol=1e-12)
    out = O.forward(x, mask, P, h, O.MASK_QUERY_KEY)
    for i in range(N):     # query j = i0 keeps only k_star in every row i
        ref = F.linear(g[0, i, i0] * v[0, i, k_star], _t(P["Wo"]), _t(P["bo"])).numpy()
        np.testing.assert_allclose(out[0, i, i0], ref, rtol=0, atol=1e-12)


def pin_zero_query_weights():
    """Wq = 0: logits are the pair bias alone, so p[t, j, :] =
    softmax(bias[b, t, j, :]) for every row i (bias from torch's linear), and
    out[b, i, j] = Wo (g * sum_k p[t, j, k] v[b, i, k]) + bo."""
    B, N, D, h = 1, 5, 8, 4
    x, _, P = _inputs(B, N, D, h, seed=16)
    P["Wq"] = np.zeros_like(P["Wq"])
    bias = F.linear(_lib_ln(x, P), _t(P["Wb"])).permute(0, 3, 1, 2)     # (B, h, j, k)
    ref = torch.softmax(bias[0], dim=-1).numpy()
    ones = np.ones((B, N, N), np.int32)
    xn = _lib_ln(x, P)
    g = torch.sigmoid(F.linear(xn, _t(P["Wg"]), _t(P["bg"])))
    v = F.linear(xn, _t(P["Wv"]))
    d = D // h
    for mode in (O.MASK_ROW_KEY, O.MASK_QUERY_KEY):
        out = O.forward(x, ones, P, h, mode)
        for i in range(N):
            p = O.attention_probs(x, ones, P, h, 0, i, mode)
            np.testing.assert_allclose(p, ref, rtol=0, atol=1e-12)
            o = torch.cat([_t(ref[t]) @ v[0, i, :, t * d:(t + 1) * d] for t in range(h)], dim=1)
            want = F.linear(g[0, i] * o, _t(P["Wo"]), _t(P["bo"])).numpy()
            np.testing.assert_allclose(out[0, i], want, rtol=0, atol=1e-12)


def pin_mean_of_kept_values():
    """Wq = Wk = Wb = 0: all logits are 0, so o is the mean of v over the kept
    keys, and over all N keys on a fully masked row (-1e9 replacement)."""
    B, N, D, h = 1, 6, 8, 2
    x, _, P = _inputs(B, N, D, h, seed=17)
    for k in ("Wq", "Wk", "Wb"):
        P[k] = np.zeros_like(P[k])
    mask = np.ones((B, N, N), np.int32)
    mask[0, 1, [0, 3]] = 0
    mask[0, 5, :] = 0
    xn = _lib_ln(x, P)
    g = torch.sigmoid(F.linear(xn, _t(P["Wg"]), _t(P["bg"])))
    v = F.linear(xn, _t(P["Wv"]))
    out = O.forward(x, mask, P, h, O.MASK_ROW_KEY)
    for i in range(N):
        kept = [k for k in range(N) if mask[0, i, k]] or list(range(N))
        mean = v[0, i, kept].mean(dim=0)
        ref = F.linear(g[0, i] * mean[None, :], _t(P["Wo"]), _t(P["bo"])).numpy()
        np.testing.assert_allclose(out[0, i], ref, rtol=0, atol=1e-12)


def pin_zero_value_weights():
    """Wv = 0: o = 0, so out = bo everywhere."""
    x, mask, P = _inputs(1, 4, 8, 2, seed=18)
    P["Wv"] = np.zeros_like(P["Wv"])
    out = O.forward(x, mask, P, 2)
    np.testing.assert_allclose(out, np.broadcast_to(P["bo"], out.shape), rtol=0, atol=1e-15)


def pin_torch_library_module():
    """Tiny shapes: the oracle equals the forward op list assembled from torch
    library routines (layer_norm, linear, scaled_dot_product_attention)."""
    for N in (1, 2, 3, 5):
        for h in (1, 2, 4):
            x, mask, P = _inputs(2, N, 8, h, seed=100 + 10 * N + h)
            for mode in (O.MASK_ROW_KEY, O.MASK_QUERY_KEY):
                np.testing.assert_allclose(O.forward(x, mask, P, h, mode),
                                           TLM.forward(x, mask, P, h, mode),
                                           rtol=0, atol=1e-12)


def pin_hand_worked_example():
    """The 2 x 2 grid of golden/hand_worked_2x2.json, derived by hand there:
    x_hat[r,c] = s[r][c] * c0 * (1, -1) with c0 = 1/sqrt(1 + 1e-5),
    l[j,k] = sqrt(2) c0^2 s[i][j] s[i][k] + c0 s[j][k],
    out[i,j] = 0.5 * sum_k softmax_k(l[j,:]) s[i][k] c0 (1, -1)."""
    with open(os.path.join(GOLDEN, "hand_worked_2x2.json")) as f:
        ex = json.load(f)
    s = ex["signs"]
    x = np.array([[[[s[r][c], -s[r][c]] for c in range(2)] for r in range(2)]], np.float64)
    P = {k: np.array(v, np.float64) for k, v in ex["params"].items()}
    out = O.forward(x, None, P, 1)
    c0 = 1.0 / math.sqrt(1.0 + 1e-5)
    for i in range(2):
        for j in range(2):
            l = [math.sqrt(2) * c0 * c0 * s[i][j] * s[i][k] + c0 * s[j][k] for k in range(2)]
            z = sum(math.exp(a) for a in l)
            o0 = sum(math.exp(l[k]) / z * s[i][k] * c0 for k in range(2))
            np.testing.assert_allclose(out[0, i, j], [0.5 * o0, -0.5 * o0], rtol=0, atol=1e-14)


def pin_hand_worked_example_ending():
    """The same 2 x 2 grid through the ending node, derived by hand in the
    fixture: cell (i, j) attends along column j,
    l[k] = sqrt(2) c0^2 s[i][j] s[k][j] + c0 s[k][i],
    out[i,j] = 0.5 * sum_k softmax_k(l) s[k][j] c0 (1, -1). The signs are not
    symmetric, so this differs from the starting node's result."""
    with open(os.path.join(GOLDEN, "hand_worked_2x2.json")) as f:
        ex = json.load(f)
    s = ex["signs"]
    x = np.array([[[[s[r][c], -s[r][c]] for c in range(2)] for r in range(2)]], np.float64)
    P = {k: np.array(v, np.float64) for k, v in ex["params"].items()}
    out = O.forward_ending(x, None, P, 1)
    c0 = 1.0 / math.sqrt(1.0 + 1e-5)
    for i in range(2):
        for j in range(2):
            l = [math.sqrt(2) * c0 * c0 * s[i][j] * s[k][j] + c0 * s[k][i] for k in range(2)]
            z = sum(math.exp(a) for a in l)
            o0 = sum(math.exp(l[k]) / z * s[k][j] * c0 for k in range(2))
            np.testing.assert_allclose(out[0, i, j], [0.5 * o0, -0.5 * o0], rtol=0, atol=1e-14)
    assert np.max(np.abs(out - O.forward(x, None, P, 1))) > 1e-2


# --------------------------------------------------------- ending-node pins

def _swap(a):
    """Exchange the two node axes of a (B, N, N, ...) array."""
    return np.swapaxes(a, 1, 2)


def pin_ending_is_module_on_swapped_grid():
    """The ending node is the starting-node module on the grid with its node
    axes exchanged: forward_ending(x, m) = T(module(T(x), T(m))), the module
    here being the torch-library statement of the op list (tiny shapes; the
    diagonal of the mask is kept so that every row and column keeps a key)."""
    for N in (1, 2, 3, 5):
        for h in (1, 2, 4):
            x, mask, P = _inputs(2, N, 8, h, seed=300 + 10 * N + h)
            mask = mask.copy()
            for r in range(N):
                mask[:, r, r] = 1
            for mode in (O.MASK_ROW_KEY, O.MASK_QUERY_KEY):
                want = _swap(TLM.forward(_swap(x), _swap(mask), P, h, mode))
                np.testing.assert_allclose(O.forward_ending(x, mask, P, h, mode), want,
                                           rtol=0, atol=1e-12)


def pin_ending_n1_closed_form():
    """N = 1: the ending node has the same closed form as the starting node."""
    for mode in (O.MASK_ROW_KEY, O.MASK_QUERY_KEY):
        x, _, P = _inputs(2, 1, 8, 2, seed=31)
        mask = np.zeros((2, 1, 1), np.int32)
        xn = _lib_ln(x, P)
        g = torch.sigmoid(F.linear(xn, _t(P["Wg"]), _t(P["bg"])))
        ref = F.linear(g * F.linear(xn, _t(P["Wv"])), _t(P["Wo"]), _t(P["bo"])).numpy()
        np.testing.assert_allclose(O.forward_ending(x, mask, P, 2, mode), ref, rtol=0, atol=1e-12)


def pin_ending_single_kept_key():
    """Row-key reading: a column j0 whose mask column pair_mask[b, :, j0] keeps
    only k* gives o[b, i, j0] = v[b, k*, j0] for every query i. Query-key
    reading: a query i0 whose column pair_mask[b, :, i0] keeps only k* gives
    o[b, i0, j] = v[b, k*, j] in every column j."""
    B, N, D, h = 1, 6, 8, 2
    x, _, P = _inputs(B, N, D, h, seed=32)
    xn = _lib_ln(x, P)
    g = torch.sigmoid(F.linear(xn, _t(P["Wg"]), _t(P["bg"])))
    v = F.linear(xn, _t(P["Wv"]))
    j0, k_star = 1, 4
    mask = np.ones((B, N, N), np.int32)
    mask[0, :, j0] = 0
    mask[0, k_star, j0] = 1
    out = O.forward_ending(x, mask, P, h, O.MASK_ROW_KEY)
    for i in range(N):
        ref = F.linear(g[0, i, j0] * v[0, k_star, j0], _t(P["Wo"]), _t(P["bo"])).numpy()
        np.testing.assert_allclose(out[0, i, j0], ref, rtol=0, atol=1e-12)
    out = O.forward_ending(x, mask, P, h, O.MASK_QUERY_KEY)
    for j in range(N):     # query i = j0 keeps only k_star in every column j
        ref = F.linear(g[0, j0, j] * v[0, k_star, j], _t(P["Wo"]), _t(P["bo"])).numpy()
        np.testing.assert_allclose(out[0, j0, j], ref, rtol=0, atol=1e-12)


def pin_ending_zero_query_weights():
    """Wq = 0, nothing masked: the ending-node weights of query i are
    softmax_k(bias[b, t, k, i]) in every column j (bias from torch's linear),
    so out[b, i, j] = Wo (g * sum_k p[t, i, k] v[b, k, j]) + bo."""
    B, N, D, h = 1, 5, 8, 4
    x, _, P = _inputs(B, N, D, h, seed=33)
    P["Wq"] = np.zeros_like(P["Wq"])
    xn = _lib_ln(x, P)
    bias = F.linear(xn, _t(P["Wb"])).permute(0, 3, 1, 2)          # (B, h, r, c)
    p = torch.softmax(bias[0].transpose(1, 2), dim=-1)             # [t, i, k] over k
    g = torch.sigmoid(F.linear(xn, _t(P["Wg"]), _t(P["bg"])))
    v = F.linear(xn, _t(P["Wv"]))
    d = D // h
    ones = np.ones((B, N, N), np.int32)
    for mode in (O.MASK_ROW_KEY, O.MASK_QUERY_KEY):
        out = O.forward_ending(x, ones, P, h, mode)
        for j in range(N):
            o = torch.cat([p[t] @ v[0, :, j, t * d:(t + 1) * d] for t in range(h)], dim=1)
            want = F.linear(g[0, :, j] * o, _t(P["Wo"]), _t(P["bo"])).numpy()
            np.testing.assert_allclose(out[0, :, j], want, rtol=0, atol=1e-12)


PINS = {f.__name__: f for f in (
    pin_n1_closed_form, pin_rows_sum_to_one, pin_all_ones_mask_is_no_mask,
    pin_relabelling_equivariance, pin_single_kept_key, pin_zero_query_weights,
    pin_mean_of_kept_values, pin_zero_value_weights, pin_torch_library_module,
    pin_hand_worked_example, pin_hand_worked_example_ending,
    pin_ending_is_module_on_swapped_grid, pin_ending_n1_closed_form,
    pin_ending_single_kept_key, pin_ending_zero_query_weights)}


@pytest.mark.parametrize("name", list(PINS))
def test_pin_holds(name):
    PINS[name]()


# ------------------------------------------------------------- planted mistakes

def _ln_wrong_axis(x, gamma, beta, eps=O.LN_EPS):
    mu = x.mean(axis=-2, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-2, keepdims=True)
    return gamma * (x - mu) / np.sqrt(var + eps) + beta


def _ln_unbiased(x, gamma, beta, eps=O.LN_EPS):
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).sum(axis=-1, keepdims=True) / (x.shape[-1] - 1)
    return gamma * (x - mu) / np.sqrt(var + eps) + beta


def _bias_transposed(bc):
    return np.transpose(bc, (0, 3, 2, 1))


def _bias_missing(bc):
    return np.zeros(np.transpose(bc, (0, 3, 1, 2)).shape)


def _keep_wrong_axis(pair_mask, b, i, mode):
    return None if pair_mask is None else pair_mask[b] != 0


def _logits_no_scale(q_i, k_i, bias_bt, keep, t, d):
    l = q_i[:, t * d:(t + 1) * d] @ k_i[:, t * d:(t + 1) * d].T + bias_bt
    return l if keep is None else np.where(keep, l, O.MASKED_LOGIT)


def _logits_half_query(q_i, k_i, bias_bt, keep, t, d):
    qh = q_i[:, t * d:(t + 1) * d].copy()
    qh[:, d // 2:] = 0.0
    l = qh @ k_i[:, t * d:(t + 1) * d].T / np.sqrt(d) + bias_bt
    return l if keep is None else np.where(keep, l, O.MASKED_LOGIT)


def _logits_neg_inf(q_i, k_i, bias_bt, keep, t, d):
    l = q_i[:, t * d:(t + 1) * d] @ k_i[:, t * d:(t + 1) * d].T / np.sqrt(d) + bias_bt
    with np.errstate(invalid="ignore"):
        return l if keep is None else np.where(keep, l, -np.inf)


def _softmax_wrong_axis(l):
    m = l.max(axis=-2, keepdims=True)
    e = np.exp(l - m)
    return e / e.sum(axis=-2, keepdims=True)


def _outproj_one_value(g_i, o_i, params):
    a = g_i * o_i
    return params["Wo"].sum(axis=1)[None, :] * a[:, :1] + params["bo"]


def _project_gate_no_bias(x_hat, params):
    q, k, v, _, bc = _REAL["project"](x_hat, params)
    return q, k, v, O.sigmoid(O.linear(x_hat, params["Wg"])), bc


def _row_attention_value_head_shift(q_i, k_i, v_i, bias_b, keep, h):
    return _REAL["row_attention"](q_i, k_i, np.roll(v_i, v_i.shape[1] // h, axis=1),
                                  bias_b, keep, h)


def _forward_rows_bias_of_row_i(x, pair_mask, params, h, rows, mask_mode=O.MASK_ROW_KEY):
    x = np.asarray(x, np.float64)
    P = {k: np.asarray(v, np.float64) for k, v in params.items()}
    B, N, _, D = x.shape
    xa = O.layer_norm(x, P["gamma"], P["beta"])
    bias = O.bias_plane(O.linear(xa, P["Wb"]))
    out = np.empty((len(rows), N, D))
    for n, (b, i) in enumerate(rows):
        q_i, k_i, v_i, g_i, _ = O.project(xa[b, i], P)
        wrong = np.broadcast_to(bias[b][:, i:i + 1, :], bias[b].shape)   # bias[b,t,i,k]
        o_i = O.row_attention(q_i, k_i, v_i, wrong, O.keep_matrix(pair_mask, b, i, mask_mode), h)
        out[n] = O.output_projection(g_i, o_i, P)
    return out


def _column_bias_untransposed(bias_b):
    return bias_b


def _column_keep_of_row(pair_mask, b, j, mode):
    return _REAL["keep_matrix"](pair_mask, b, j, mode)


def _forward_ending_row_cells(x, pair_mask, params, h, cols, mask_mode=O.MASK_ROW_KEY):
    x = np.asarray(x, np.float64)
    P = {k: np.asarray(v, np.float64) for k, v in params.items()}
    B, N, _, D = x.shape
    xa = O.layer_norm(x, P["gamma"], P["beta"])
    bias = O.bias_plane(O.linear(xa, P["Wb"]))
    out = np.empty((len(cols), N, D))
    for n, (b, j) in enumerate(cols):
        q_j, k_j, v_j, g_j, _ = O.project(xa[b, j, :], P)          # row j, not column j
        o_j = O.row_attention(q_j, k_j, v_j, O.column_bias(bias[b]),
                              O.column_keep(pair_mask, b, j, mask_mode), h)
        out[n] = O.output_projection(g_j, o_j, P)
    return out


_REAL = {n: getattr(O, n) for n in ("project", "row_attention", "keep_matrix")}

MISTAKES = [
    # (oracle attribute, wrong stand-in, the pin that must catch it)
    ("layer_norm", _ln_wrong_axis, "pin_n1_closed_form"),
    ("layer_norm", _ln_unbiased, "pin_n1_closed_form"),
    ("bias_plane", _bias_transposed, "pin_zero_query_weights"),
    ("bias_plane", _bias_missing, "pin_zero_query_weights"),
    ("forward_rows", _forward_rows_bias_of_row_i, "pin_zero_query_weights"),
    ("keep_matrix", _keep_wrong_axis, "pin_single_kept_key"),
    ("head_logits", _logits_no_scale, "pin_torch_library_module"),
    ("head_logits", _logits_no_scale, "pin_hand_worked_example"),
    ("head_logits", _logits_half_query, "pin_torch_library_module"),
    ("head_logits", _logits_neg_inf, "pin_mean_of_kept_values"),
    ("softmax_last", _softmax_wrong_axis, "pin_rows_sum_to_one"),
    ("output_projection", _outproj_one_value, "pin_n1_closed_form"),
    ("project", _project_gate_no_bias, "pin_n1_closed_form"),
    ("row_attention", _row_attention_value_head_shift, "pin_single_kept_key"),
    ("column_bias", _column_bias_untransposed, "pin_ending_zero_query_weights"),
    ("column_bias", _column_bias_untransposed, "pin_ending_is_module_on_swapped_grid"),
    ("column_keep", _column_keep_of_row, "pin_ending_single_kept_key"),
    ("forward_ending_columns", _forward_ending_row_cells, "pin_ending_is_module_on_swapped_grid"),
    ("forward_ending_columns", _forward_ending_row_cells, "pin_ending_single_kept_key"),
]


@pytest.mark.parametrize("attr,wrong,pin", MISTAKES,
                         ids=[f"{a}:{w.__name__}->{p}" for a, w, p in MISTAKES])
def test_planted_mistake_is_caught(monkeypatch, attr, wrong, pin):
    monkeypatch.setattr(O, attr, wrong)
    with pytest.raises(AssertionError):
        with np.errstate(all="ignore"):
            PINS[pin]()
