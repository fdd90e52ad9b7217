"""The forward pass assembled from PyTorch library routines, in float64 on the CPU.

A second statement of the method, written from a different description than the
oracle: the oracle follows per-index formulas, while this one follows the
tensor-op sequence of the forward op list on the POPCORNBENCH page
"Kimi-K2.6 l2_p6" (steps 1-18: reshape, view, transpose, broadcast) and hands the
attention step to ``torch.nn.functional.scaled_dot_product_attention`` and the
normalisation to ``torch.nn.functional.layer_norm``. It is used only to pin the
oracle on tiny inputs.

The mask enters SDPA as an additive float term (-1e9 on dropped keys), which
equals the oracle's replacement by -1e9 on every softmax row that keeps at least
one key; callers use masks where every row keeps one.
"""
import math

import torch
import torch.nn.functional as F


def forward(x, pair_mask, params, h, mask_mode=0):
    t = lambda a: torch.as_tensor(a, dtype=torch.float64)
    x = t(x)
    P = {k: t(v) for k, v in params.items()}
    B, N, _, D = x.shape
    d = D // h
    xn = F.layer_norm(x, (D,), P["gamma"], P["beta"], eps=1e-5)               # step 1
    g = torch.sigmoid(F.linear(xn, P["Wg"], P["bg"]))                        # step 2
    bias = F.linear(xn, P["Wb"]).permute(0, 3, 1, 2)                         # step 3
    x_flat = xn.reshape(B * N, N, D)                                         # step 4
    q = F.linear(x_flat, P["Wq"]).view(B * N, N, h, d).transpose(1, 2)      # step 5
    k = F.linear(x_flat, P["Wk"]).view(B * N, N, h, d).transpose(1, 2)      # step 6
    v = F.linear(x_flat, P["Wv"]).view(B * N, N, h, d).transpose(1, 2)      # step 7
    add = bias.unsqueeze(1).expand(B, N, h, N, N)                            # steps 9-10
    if pair_mask is not None:
        m = torch.as_tensor(pair_mask) != 0
        if mask_mode == 0:      # key k of row i: pair_mask[b, i, k]
            keep = m.view(B, N, 1, 1, N)
        else:                   # query j, key k: pair_mask[b, j, k] (steps 11-12)
            keep = m.unsqueeze(1).unsqueeze(2)
        add = add + torch.where(keep, 0.0, -1e9).to(torch.float64)
    add = add.reshape(B * N, h, N, N)                                        # step 13
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=add,               # steps 8, 14-16
                                       scale=1.0 / math.sqrt(d))
    o = o.transpose(1, 2).reshape(B, N, N, D)
    return F.linear(g * o, P["Wo"], P["bo"]).numpy()                         # steps 17-18
