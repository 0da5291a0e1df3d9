"""Brute-force per-token MoE forward in pure Python (tiny inputs only).

TEST INFRASTRUCTURE (same rule as oracle/moe_oracle.py).  It pins the fp64
oracle: it follows the per-token reading of Algorithm 2 of "MoE 分布式推理基础
（基于 vLLM）" §1.2 -- for one token, score every expert, keep the K best,
weight each chosen expert's SwiGLU output and add -- with scalar loops and
the math module only: no numpy, no matrix products, no permutation.  A
layout, gather or combine mistake in the oracle cannot be reproduced here.
"""
from __future__ import annotations

import math


def _row(a, i):
    return [float(v) for v in a[i]]


def token_forward(x_row, w_gate, bias, w13, w2, K, norm_topk_prob):
    """One token.  x_row: H floats; w_gate[h][e]; bias[e] or None;
    w13[e][h][j] (j < I gate, j >= I up); w2[e][i][c].
    Returns (experts, weights, y_row)."""
    H = len(x_row)
    E = len(w_gate[0])
    I = len(w2[0])
    scores = []
    for e in range(E):
        s = 0.0
        for hh in range(H):
            s += x_row[hh] * float(w_gate[hh][e])
        if bias is not None:
            s += float(bias[e])
        scores.append(s)
    experts = sorted(range(E), key=lambda e: (-scores[e], e))[:K]
    top = max(scores)
    z = [math.exp(s - top) for s in scores]
    total = sum(z)
    weights = [z[e] / total for e in experts]
    if norm_topk_prob:
        ws = sum(weights)
        weights = [w / ws for w in weights]
    y = [0.0] * H
    for w, e in zip(weights, experts):
        act = []
        for i in range(I):
            g = 0.0
            u = 0.0
            for hh in range(H):
                g += x_row[hh] * float(w13[e][hh][i])
                u += x_row[hh] * float(w13[e][hh][I + i])
            sig = 1.0 / (1.0 + math.exp(-g)) if g > -700 else 0.0
            act.append(g * sig * u)
        for c in range(H):
            acc = 0.0
            for i in range(I):
                acc += act[i] * float(w2[e][i][c])
            y[c] += w * acc
    return experts, weights, y


def moe_forward_brute(x, w_gate, bias, w13, w2, K, norm_topk_prob, tokens=None):
    """Per-token loop over `tokens` (default: all).  Returns lists
    (experts, weights, y) indexed like `tokens`."""
    idx = range(len(x)) if tokens is None else tokens
    out_e, out_w, out_y = [], [], []
    for t in idx:
        e, w, y = token_forward(_row(x, t), w_gate, bias, w13, w2, K, norm_topk_prob)
        out_e.append(e)
        out_w.append(w)
        out_y.append(y)
    return out_e, out_w, out_y
