"""Oracle: a plain, slow fp64 CPU statement of starting-node triangular
self-attention (forward pass, eval mode).

TEST INFRASTRUCTURE. Only the test-suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run this module. The product
path (the CUDA library and its Python binding) never calls it, and this module
imports nothing from the product package.

Sources (POPCORNBENCH transcripts, triangular self-attention):
  [P1] "FW-GLM-5-1 l2_p6" -- the quoted reference ``Model.forward``.
  [P2] "Kimi-K2.6 l2_p6"  -- the 18-step forward op list, the layer
       definitions (which ``nn.Linear`` carries a bias) and the kernel sketches.

Everything is evaluated in float64 from the exact input values (bf16 inputs
arrive already rounded, as float32 arrays). Matrix products use numpy's
``@`` as a library step; nothing is blocked, fused or reordered beyond the
definition below.

Definition (cell (b, r, c) of the pair grid; d = D / h; head t owns channels
t*d .. t*d+d-1):

    x_hat[b,r,c]   = gamma * (x - mean) / sqrt(var + 1e-5) + beta   (biased var over D)
    q, k, v        = Wq x_hat, Wk x_hat, Wv x_hat                   (no bias)
    g              = sigmoid(Wg x_hat + bg)
    bias[b,t,r,c]  = (Wb x_hat[b,r,c])[t]                           (no bias)
    for each (b, i, t, j):
      l_k  = q[b,i,j,t] . k[b,i,k,t] / sqrt(d) + bias[b,t,j,k]     (k = 0..N-1)
      l_k := -1e9 where the mask drops key k                       (replacement)
      p    = softmax over k of l
      o[b,i,j,t] = sum_k p_k v[b,i,k,t]
    out[b,i,j]     = Wo (g[b,i,j] * o[b,i,j]) + bo                  (dropout = identity)

Readings where the pages are silent or disagree:
  * Mask axis. The quoted code broadcasts ``pair_mask`` over rows i, so key k
    of query j is dropped when pair_mask[b, j, k] == 0 (MASK_QUERY_KEY). The
    task statement drops key k of row i when pair_mask[b, i, k] == 0
    (MASK_ROW_KEY, the default). Both are implemented.
  * Masked logits are replaced by -1e9 ([P2] kernel sketch) rather than filled
    with -inf ([P1] ``masked_fill``): a fully masked softmax row then gets the
    uniform weight 1/N instead of NaN.
  * Dropout is the identity (eval mode, [P2] discussion of ``nn.Dropout``).
  * Any nonzero mask entry keeps the key.
  * Ending-node variant. The pages name only the starting-node module. Its
    counterpart is read as the same module applied to the grid with its two
    node axes exchanged: out_end = T(out_start(T(x), T(pair_mask))), T swapping
    the two N axes. Written out per output cell (b, i, j), the softmax then
    runs along column j:
        l_k = q[b,i,j,t] . k[b,k,j,t] / sqrt(d) + bias[b,t,k,i]
        o[b,i,j,t] = sum_k p_k v[b,k,j,t]
    and key k is dropped when pair_mask[b,k,j] == 0 (MASK_ROW_KEY) or
    pair_mask[b,k,i] == 0 (MASK_QUERY_KEY). ``forward_ending`` computes this
    per column from the formula, not through the transposes.
"""
from __future__ import annotations

import numpy as np

MASK_ROW_KEY = 0
MASK_QUERY_KEY = 1
MASKED_LOGIT = -1e9
LN_EPS = 1e-5


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def layer_norm(x, gamma, beta, eps=LN_EPS):
    """[P1] ``self.layer_norm(pair_repr)``; [P2] op list step 1. Over the last
    axis, biased variance, eps inside the square root."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return gamma * (x - mu) / np.sqrt(var + eps) + beta


def linear(x, W, b=None):
    """``nn.Linear``: y = x W^T (+ b); W is (out_features, in_features)."""
    y = x @ W.T
    return y if b is None else y + b


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def project(x_hat, params):
    """[P2] op list steps 2, 3, 5-7 and the layer definitions: q, k, v and the
    pair-bias projection carry no bias; the gate does. Returns q, k, v, g of
    shape (..., D) and the per-cell bias of shape (..., h)."""
    q = linear(x_hat, params["Wq"])
    k = linear(x_hat, params["Wk"])
    v = linear(x_hat, params["Wv"])
    g = sigmoid(linear(x_hat, params["Wg"], params["bg"]))
    bias_cells = linear(x_hat, params["Wb"])
    return q, k, v, g, bias_cells


def bias_plane(bias_cells):
    """[P1] ``bias_proj(x).permute(0, 3, 1, 2)``: (B, N, N, h) -> (B, h, N, N)."""
    return np.transpose(bias_cells, (0, 3, 1, 2))


def keep_matrix(pair_mask, b, i, mask_mode):
    """Boolean keep[j, k] for softmax row (b, i): which keys each query sees.

    MASK_ROW_KEY:   keep[j, k] = pair_mask[b, i, k] != 0 (same for every j).
    MASK_QUERY_KEY: keep[j, k] = pair_mask[b, j, k] != 0 ([P1] broadcast of
                    ``pair_mask.unsqueeze(1).unsqueeze(2)`` over rows i).
    ``pair_mask=None`` keeps every key."""
    if pair_mask is None:
        return None
    N = pair_mask.shape[-1]
    if mask_mode == MASK_ROW_KEY:
        return np.broadcast_to(pair_mask[b, i, :] != 0, (N, N))
    if mask_mode == MASK_QUERY_KEY:
        return pair_mask[b] != 0
    raise ValueError(f"unknown mask mode {mask_mode}")


def softmax_last(l):
    """Softmax over the last axis (keys), [P2] op list step 14."""
    m = l.max(axis=-1, keepdims=True)
    e = np.exp(l - m)
    return e / e.sum(axis=-1, keepdims=True)


def head_logits(q_i, k_i, bias_bt, keep, t, d):
    """[P2] op list steps 8-12 for one (b, i, head t): (N, N) logits l[j, k]."""
    qh = q_i[:, t * d:(t + 1) * d]
    kh = k_i[:, t * d:(t + 1) * d]
    l = (qh @ kh.T) / np.sqrt(d) + bias_bt
    if keep is not None:
        l = np.where(keep, l, MASKED_LOGIT)
    return l


def row_attention(q_i, k_i, v_i, bias_b, keep, h):
    """Attention of softmax row (b, i) over its N keys, all heads.

    q_i, k_i, v_i: (N, D) for cells (b, i, 0..N-1); bias_b: (h, N, N);
    keep: (N, N) or None. Returns o_i (N, D) with o[j, t*d + e] =
    sum_k p[t, j, k] v[k, t*d + e]  ([P2] op list steps 13-16)."""
    N, D = q_i.shape
    d = D // h
    o = np.empty((N, D))
    for t in range(h):
        p = softmax_last(head_logits(q_i, k_i, bias_b[t], keep, t, d))
        o[:, t * d:(t + 1) * d] = p @ v_i[:, t * d:(t + 1) * d]
    return o


def attention_probs(x, pair_mask, params, h, b, i, mask_mode=MASK_ROW_KEY):
    """Softmax weights p[t, j, k] of row (b, i): (h, N, N). For invariant tests."""
    x_hat = layer_norm(_f64(x), _f64(params["gamma"]), _f64(params["beta"]))
    P = {k: _f64(v) for k, v in params.items()}
    q, k, _, _, bc = project(x_hat, P)
    bias = bias_plane(bc)
    N, D = x.shape[1], x.shape[3]
    d = D // h
    keep = keep_matrix(pair_mask, b, i, mask_mode)
    return np.stack([softmax_last(head_logits(q[b, i], k[b, i], bias[b, t], keep, t, d))
                     for t in range(h)])


def output_projection(g_i, o_i, params):
    """[P2] op list steps 17-18: out = Wo (g * o) + bo."""
    return linear(g_i * o_i, params["Wo"], params["bo"])


def forward_rows(x, pair_mask, params, h, rows, mask_mode=MASK_ROW_KEY):
    """``out[b, i, :, :]`` for each (b, i) in ``rows``: array (len(rows), N, D).

    The bias plane needs every cell; q, k, v and g are needed only for the
    cells of the requested rows."""
    P = {k: _f64(v) for k, v in params.items()}
    B, N, _, D = x.shape
    h_out = P["Wb"].shape[0]
    # The per-cell bias, one grid row at a time (the same per-cell LayerNorm and
    # projection; only the memory held at once is bounded).
    bias_cells = np.empty((B, N, N, h_out))
    for b in range(B):
        for r in range(N):
            bias_cells[b, r] = linear(layer_norm(_f64(x[b, r]), P["gamma"], P["beta"]), P["Wb"])
    bias = bias_plane(bias_cells)
    out = np.empty((len(rows), N, D))
    for n, (b, i) in enumerate(rows):
        q_i, k_i, v_i, g_i, _ = project(layer_norm(_f64(x[b, i]), P["gamma"], P["beta"]), P)
        keep = keep_matrix(pair_mask, b, i, mask_mode)
        o_i = row_attention(q_i, k_i, v_i, bias[b], keep, h)
        out[n] = output_projection(g_i, o_i, P)
    return out


def forward(x, pair_mask, params, h, mask_mode=MASK_ROW_KEY):
    """Full forward: out (B, N, N, D) in float64. ``pair_mask=None`` = no mask."""
    B, N = x.shape[0], x.shape[1]
    rows = [(b, i) for b in range(B) for i in range(N)]
    return forward_rows(x, pair_mask, params, h, rows, mask_mode).reshape(x.shape)


# ---------------------------------------------------------------- ending node
def column_keep(pair_mask, b, j, mask_mode):
    """Boolean keep[i, k] for the ending-node softmax of column (b, j).

    MASK_ROW_KEY:   keep[i, k] = pair_mask[b, k, j] != 0 (same for every query i).
    MASK_QUERY_KEY: keep[i, k] = pair_mask[b, k, i] != 0.
    ``pair_mask=None`` keeps every key."""
    if pair_mask is None:
        return None
    N = pair_mask.shape[-1]
    if mask_mode == MASK_ROW_KEY:
        return np.broadcast_to(pair_mask[b, :, j] != 0, (N, N))
    if mask_mode == MASK_QUERY_KEY:
        return (pair_mask[b] != 0).T
    raise ValueError(f"unknown mask mode {mask_mode}")


def column_bias(bias_b):
    """Pair bias of the ending-node softmax: entry [t, i, k] (query i, key k)
    is bias[b, t, k, i]."""
    return np.transpose(bias_b, (0, 2, 1))


def forward_ending_columns(x, pair_mask, params, h, cols, mask_mode=MASK_ROW_KEY):
    """Ending node: ``out[b, :, j, :]`` for each (b, j) in ``cols``, array
    (len(cols), N, D). Column (b, j) holds the queries i (cells (b, i, j)) and
    the keys k (cells (b, k, j)) of its softmax."""
    x = _f64(x)
    P = {k: _f64(v) for k, v in params.items()}
    B, N, _, D = x.shape
    x_hat_all = layer_norm(x, P["gamma"], P["beta"])
    bias = bias_plane(linear(x_hat_all, P["Wb"]))
    out = np.empty((len(cols), N, D))
    for n, (b, j) in enumerate(cols):
        q_j, k_j, v_j, g_j, _ = project(x_hat_all[b, :, j], P)
        keep = column_keep(pair_mask, b, j, mask_mode)
        o_j = row_attention(q_j, k_j, v_j, column_bias(bias[b]), keep, h)
        out[n] = output_projection(g_j, o_j, P)
    return out


def forward_ending(x, pair_mask, params, h, mask_mode=MASK_ROW_KEY):
    """Ending-node forward: out (B, N, N, D) in float64."""
    B, N, D = x.shape[0], x.shape[1], x.shape[3]
    cols = [(b, j) for b in range(B) for j in range(N)]
    res = forward_ending_columns(x, pair_mask, params, h, cols, mask_mode)
    return res.reshape(B, N, N, D).transpose(0, 2, 1, 3)
