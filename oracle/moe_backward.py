"""fp64 CPU oracle of the MoE layer's backward pass.

TEST INFRASTRUCTURE.  Only the test suite (tests/), __graft_entry__.smoke()
and bench.py's CPU-baseline / reference arm may import or call this module.
The library under top_routing_dispatch_gb300/ never does, and this module
shares no code with it.

What it computes: the gradient of the forward of moe_oracle.moe_forward
(Algorithm 2 of "MoE 分布式推理基础（基于 vLLM）", §1.2) for an upstream
gradient dy = dL/dy, with the expert choice (the TopK indices) held fixed,
as automatic differentiation of a top-k selection does.  The pages give the
structure, not the formulas: "大模型系统中的通算融合" §6.2.4 states that in
training the backward of dispatch is a combine and the backward of combine
is a dispatch, and the DModel notes ("0. goin", §2.3, the MinimalAsyncEP
kernel table) list the backward of the top-k reduce and a routing-score
gradient next to the forward kernels.  Written out (plain calculus, float64,
no rounding):

  combine backward (a dispatch):   dY[r] = w[f] * dy[t],  dw[f] = <dy[t], Y[r]>
                                   for every pair f = t*K + k, r = inv_perm[f]
  expert backward (expert e):      dh = dY_e W2[e]^T,      dW2[e]  = h_e^T dY_e
                                   dG = dh * U * s * (1 + G (1 - s)),  s = sigmoid(G)
                                   dU = dh * G * s
                                   dX_e = [dG | dU] W13[e]^T,  dW13[e] = X_e^T [dG | dU]
  permute backward (a combine):    dx[t] = sum_k dX[inv_perm[t*K + k]]
  router backward:                 dp over the selected experts from dw (through
                                   the renormalisation when norm_topk_prob),
                                   dlogits = p * (dp - <p, dp>) (softmax),
                                   dx += dlogits W_gate^T,  dW_gate = x^T dlogits,
                                   dbias = sum_t dlogits[t]

Library primitives used as steps: numpy matmul (BLAS), exp.
"""
from __future__ import annotations

import numpy as np

from . import moe_oracle as F

F64 = np.float64


def _f64(a):
    return None if a is None else np.asarray(a, dtype=F64)


def combine_backward(dy, y_perm, w_top, inv_perm):
    """dY[r] = w[f] dy[t] and dw[f] = <dy[t], Y[r]> for f = t*K + k,
    r = inv_perm[f].  Returns (dY (nK, H), dw (n, K))."""
    dy = _f64(dy)
    w_top = _f64(w_top)
    n, K = w_top.shape
    inv = np.asarray(inv_perm).reshape(n, K)
    y_perm = _f64(y_perm)
    dY = np.zeros_like(y_perm)
    dw = np.zeros((n, K), dtype=F64)
    for k in range(K):
        dY[inv[:, k]] = w_top[:, k:k + 1] * dy
        dw[:, k] = np.einsum("th,th->t", dy, y_perm[inv[:, k]])
    return dY, dw


def expert_backward(X_e, W13_e, W2_e, dY_e):
    """Backward of one expert's SwiGLU MLP.  Returns dict(dh, dG, dU, dX,
    dW13, dW2) for the rows X_e (n_e, H) and their output gradient dY_e."""
    X_e, W13_e, W2_e, dY_e = _f64(X_e), _f64(W13_e), _f64(W2_e), _f64(dY_e)
    I = W13_e.shape[1] // 2
    gate_up = X_e @ W13_e
    G, U = gate_up[:, :I], gate_up[:, I:]
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-G))
    h = G * s * U
    dh = dY_e @ W2_e.T
    dG = dh * U * s * (1.0 + G * (1.0 - s))
    dU = dh * G * s
    dGU = np.concatenate([dG, dU], axis=1)
    return dict(h=h, dh=dh, dG=dG, dU=dU, dGU=dGU, dX=dGU @ W13_e.T, dW13=X_e.T @ dGU,
                dW2=h.T @ dY_e)


def router_backward(x, w_gate, logits, e_top, w_top, dw, norm_topk_prob):
    """Gradient through the TopK weights, the renormalisation and the
    softmax.  Returns (dlogits (n, E), dx_router (n, H), dW_gate (H, E))."""
    x, w_gate, logits = _f64(x), _f64(w_gate), _f64(logits)
    dw, w_top = _f64(dw), _f64(w_top)
    n, E = logits.shape
    p = F.softmax(logits)
    rows = np.arange(n)[:, None]
    p_sel = p[rows, e_top]
    if norm_topk_prob:
        S = p_sel.sum(axis=1, keepdims=True)
        dp_sel = (dw - (dw * w_top).sum(axis=1, keepdims=True)) / S
    else:
        dp_sel = dw
    dp = np.zeros((n, E), dtype=F64)
    dp[rows, e_top] = dp_sel
    dlogits = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    return dlogits, dlogits @ w_gate.T, x.T @ dlogits


def moe_backward(x, w_gate, bias, w13, w2, K, norm_topk_prob, dy, forced=None):
    """Forward (moe_oracle.moe_forward) then the backward for dy.  Returns
    the forward's dict extended with dY, dw, dh, dGU, dx_perm, dx_experts,
    dlogits, dx, dw_gate, dbias, dw13 (E, H, 2I), dw2 (E, I, H)."""
    fw = F.moe_forward(x, w_gate, bias, w13, w2, K, norm_topk_prob, forced=forced)
    x = _f64(x)
    n, H = x.shape
    offsets, perm, inv_perm = fw["offsets"], fw["perm"], fw["inv_perm"]
    E = len(offsets) - 1
    dY, dw = combine_backward(dy, fw["y_perm"], fw["w_top"], inv_perm)
    x_perm = F.permute(x, perm, K)
    nK = x_perm.shape[0]
    I = F._expert(w2, 0).shape[0]
    dh = np.zeros((nK, I), dtype=F64)
    dGU = np.zeros((nK, 2 * I), dtype=F64)
    dx_perm = np.zeros((nK, H), dtype=F64)
    dw13 = np.zeros((E, H, 2 * I), dtype=F64)
    dw2 = np.zeros((E, I, H), dtype=F64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        b = expert_backward(x_perm[lo:hi], F._expert(w13, e), F._expert(w2, e), dY[lo:hi])
        dh[lo:hi], dGU[lo:hi], dx_perm[lo:hi] = b["dh"], b["dGU"], b["dX"]
        dw13[e], dw2[e] = b["dW13"], b["dW2"]
    inv = np.asarray(inv_perm).reshape(n, K)
    dx_experts = dx_perm[inv].sum(axis=1)
    dlogits, dx_router, dw_gate = router_backward(x, w_gate, fw["logits"], fw["e_top"],
                                                  fw["w_top"], dw, norm_topk_prob)
    out = dict(fw)
    out.update(dY=dY, dw=dw, dh=dh, dGU=dGU, dx_perm=dx_perm, dx_experts=dx_experts,
               dlogits=dlogits, dx=dx_experts + dx_router, dw_gate=dw_gate,
               dbias=dlogits.sum(axis=0), dw13=dw13, dw2=dw2)
    return out
