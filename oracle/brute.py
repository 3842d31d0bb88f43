"""Pure-Python fp64 brute force of the multi-head attention forward pass.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``). Explicit loops over
Python floats, for tiny inputs only (a few thousand multiply-adds); it is the
second, independent implementation that pins the C oracle.

Each step follows the pages:
  * nn.Linear y = x W^T + b -- "003-Transformer" tutorial, MultiHeadedAttention
    (four nn.Linear(embedding_dim, embedding_dim)).
  * head i owns output features [i*d_k, (i+1)*d_k) -- the view(B, -1, h, d_k)
    in MultiHeadedAttention.forward.
  * scores / sqrt(d_k), masked_fill(mask == 0, -1e9), softmax over keys, P.V --
    "The Annotated Transformer", section "Attention", attention().
  * concat of heads in head order, then the fourth Linear.
"""
from __future__ import annotations

import math


def linear(x, W, b):
    """x: list of rows; W: [out][in]; b: [out] or None."""
    out = []
    for row in x:
        y = []
        for o in range(len(W)):
            acc = 0.0
            for i in range(len(row)):
                acc += row[i] * W[o][i]
            y.append(acc + (b[o] if b is not None else 0.0))
        out.append(y)
    return out


def allowed(b, i, j, causal, valid_lens, dense):
    if causal and j > i:
        return False
    if valid_lens is not None and j >= valid_lens[b]:
        return False
    if dense is not None:
        qi = 0 if len(dense[b]) == 1 else i
        if dense[b][qi][j] == 0:
            return False
    return True


def mha_forward(query, key, value, w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o, h,
                causal=False, valid_lens=None, dense=None):
    """Nested lists in, nested lists out: (out [B][Lq][d], p_attn [B][h][Lq][Lk])."""
    B = len(query)
    d = len(w_q)
    dk = d // h
    out_all, p_all = [], []
    for b in range(B):
        Q = linear(query[b], w_q, b_q)
        K = linear(key[b], w_k, b_k)
        V = linear(value[b], w_v, b_v)
        Lq, Lk = len(Q), len(K)
        ctx = [[0.0] * d for _ in range(Lq)]
        p_b = []
        for hh in range(h):
            p_h = []
            for i in range(Lq):
                s = []
                for j in range(Lk):
                    dot = 0.0
                    for c in range(dk):
                        dot += Q[i][hh * dk + c] * K[j][hh * dk + c]
                    sc = dot / math.sqrt(dk)
                    if not allowed(b, i, j, causal, valid_lens, dense):
                        sc = -1e9
                    s.append(sc)
                m = max(s)
                e = [math.exp(x - m) for x in s]
                z = sum(e)
                p = [x / z for x in e]
                p_h.append(p)
                for c in range(dk):
                    acc = 0.0
                    for j in range(Lk):
                        acc += p[j] * V[j][hh * dk + c]
                    ctx[i][hh * dk + c] = acc
            p_b.append(p_h)
        out_all.append(linear(ctx, w_o, b_o))
        p_all.append(p_b)
    return out_all, p_all


def ffn_forward(x, w_1, b_1, w_2, b_2):
    """Position-wise FFN, nested lists: max(0, x W_1^T + b_1) W_2^T + b_2 per row
    ("003-Transformer" tutorial, feed-forward layer)."""
    hid = linear(x, w_1, b_1)
    hid = [[v if v > 0.0 else 0.0 for v in row] for row in hid]
    return linear(hid, w_2, b_2)
