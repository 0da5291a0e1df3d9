"""fp64 CPU oracle of the single-card MoE layer forward.

TEST INFRASTRUCTURE.  Only the test suite (tests/), __graft_entry__.smoke()
and bench.py's CPU-baseline / reference arm may import or call this module.
The library under top_routing_dispatch_gb300/ never does, and this module
shares no code with it.

What it computes: Algorithm 2 ("Single-GPU MoE Forward (OlmoeExperts)") of
the page "MoE 分布式推理基础（基于 vLLM）", §1.2 "MoE Forward", together with
the router's optional renormalisation shown in the same section (when
norm_topk_prob is set, the K selected probabilities are divided by their
sum).  All
arithmetic is float64 on exactly upcast inputs; nothing is rounded to the
GPU's storage types.  Library primitives used as steps: numpy matmul (BLAS),
exp, and a stable argsort.

Readings taken where the page leaves a step open (each is listed with its
reason in the design notes):
  * TopK order: slots sorted by descending logit; an exact tie goes to the
    lower expert index.  Selecting on logits gives the same order as
    selecting on p = softmax(logits) (softmax is monotone).
  * Skewed workload: a per-expert bias is added to the router logits.
  * Dispatch layout: the (token, slot) pairs are flattened to f = t*K + k and
    stably sorted by expert, i.e. ascending f inside each expert -- the order
    that the `moe_align_block_size` worked example of §2.3 prints.
  * SwiGLU: gate = first I columns of X_e·W13[e], up = last I columns (the
    2I outputs are split in two halves in §1.2, "SwiGLU expert 的两段 GEMM").
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def _f64(a):
    return None if a is None else np.asarray(a, dtype=F64)


def _expert(src, e):
    """Expert e's weight slice as float64; `src` is an (E, ...) array or a
    callable e -> array (lets a caller stream one expert at a time)."""
    w = src(e) if callable(src) else src[e]
    return np.asarray(w, dtype=F64)


# --------------------------------------------------------------------------
# Router: Algorithm 2 steps 1-3 (+ renormalisation of OlmoeTopKRouter)
# --------------------------------------------------------------------------

def router_logits(x, w_gate, bias=None):
    """Step 1: l = x · W_gate, shape (n, E).  `bias` (E,) is added per expert
    when given (skewed-routing workload)."""
    logits = _f64(x) @ _f64(w_gate)
    if bias is not None:
        logits = logits + _f64(bias)[None, :]
    return logits


def softmax(logits):
    """Step 2: p = softmax(l) along the expert axis (max-shifted exp)."""
    logits = _f64(logits)
    m = np.max(logits, axis=1, keepdims=True)
    z = np.exp(logits - m)
    return z / np.sum(z, axis=1, keepdims=True)


def topk(logits, K, norm_topk_prob):
    """Step 3: (w_top, e_top) = TopK(p, K), then w_top /= sum(w_top) when
    norm_topk_prob.  Returns e_top (n, K) int64 in descending-logit order
    (ties: lower expert first) and w_top (n, K) float64."""
    logits = _f64(logits)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :K]
    p = softmax(logits)
    w_top = np.take_along_axis(p, order, axis=1)
    if norm_topk_prob:
        w_top = w_top / np.sum(w_top, axis=1, keepdims=True)
    return order.astype(np.int64), w_top


def weights_for(logits, e_top, norm_topk_prob):
    """w_top for a given expert choice: p at the chosen experts, renormalised
    when norm_topk_prob (used when a near-tie token's choice is imposed)."""
    p = softmax(logits)
    w = np.take_along_axis(p, np.asarray(e_top, dtype=np.int64), axis=1)
    if norm_topk_prob:
        w = w / np.sum(w, axis=1, keepdims=True)
    return w


def near_tie_tokens(logits, K, gap=1e-6):
    """Boolean mask of tokens whose top-(K+1) sorted logits have an adjacent
    gap below `gap` (their TopK order or membership is decided by rounding).
    Two equal infinite logits count as a tie."""
    logits = _f64(logits)
    E = logits.shape[1]
    m = min(K + 1, E)
    s = -np.sort(-logits, axis=1)[:, :m]
    if m < 2:
        return np.zeros(logits.shape[0], dtype=bool)
    with np.errstate(invalid="ignore"):
        d = s[:, :-1] - s[:, 1:]
    return np.any(~(d >= gap), axis=1)


# --------------------------------------------------------------------------
# Dispatch layout: Algorithm 2 steps 4-5 (hit counts n_e, sets I_e)
# --------------------------------------------------------------------------

def dispatch_layout(e_top, E):
    """counts[e] = n_e = #{(i,k): e_top[i,k] = e}; offsets = exclusive scan
    (E+1 entries, offsets[E] = n*K); perm[r] = flat index f = i*K + k of the
    r-th pair after a stable sort by expert; inv_perm[perm[r]] = r."""
    flat = np.asarray(e_top, dtype=np.int64).reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    perm = np.argsort(flat, kind="stable").astype(np.int64)
    inv_perm = np.empty_like(perm)
    inv_perm[perm] = np.arange(perm.size, dtype=np.int64)
    return counts, offsets, perm, inv_perm


def padded_block_layout(counts, offsets, perm, block_m, pad):
    """The block-padded form of the layout printed by `moe_align_block_size`
    (§2.3): each expert's run of flat ids is padded with `pad` to a multiple of
    block_m; expert_ids names the expert of every block."""
    sorted_ids, expert_ids = [], []
    for e, c in enumerate(counts):
        if c == 0:
            continue
        seg = list(perm[offsets[e]:offsets[e + 1]])
        nb = -(-int(c) // block_m)
        seg += [pad] * (nb * block_m - int(c))
        sorted_ids += seg
        expert_ids += [e] * nb
    return sorted_ids, expert_ids, len(sorted_ids)


# --------------------------------------------------------------------------
# Gather, experts, combine: Algorithm 2 steps 7-11
# --------------------------------------------------------------------------

def permute(x, perm, K):
    """Step 7 for all experts at once: x_perm[r] = x[perm[r] // K]."""
    return _f64(x)[np.asarray(perm) // K]


def expert_up(X_e, W13_e):
    """Step 8: G_e = SiLU(X_e W13[:, :I]) * (X_e W13[:, I:]), with
    SiLU(g) = g * sigmoid(g) = g / (1 + exp(-g))."""
    I = W13_e.shape[1] // 2
    gate_up = X_e @ W13_e
    gate, up = gate_up[:, :I], gate_up[:, I:]
    with np.errstate(over="ignore"):
        return gate / (1.0 + np.exp(-gate)) * up


def expert_down(G_e, W2_e):
    """Step 9: Y_e = G_e W2."""
    return G_e @ W2_e


def swiglu_expert(X_e, W13_e, W2_e):
    """Steps 8-9 for one expert.  Returns (G_e, Y_e)."""
    G_e = expert_up(X_e, W13_e)
    return G_e, expert_down(G_e, W2_e)


def grouped_swiglu(x_perm, offsets, w13, w2):
    """Steps 4-9 over every expert with n_e > 0 (empty experts are skipped,
    step 6).  Returns h (nK, I) and y_perm (nK, H) in the permuted order."""
    x_perm = _f64(x_perm)
    E = len(offsets) - 1
    nK, H = x_perm.shape
    h = None
    y_perm = np.zeros((nK, H), dtype=F64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        G_e, Y_e = swiglu_expert(x_perm[lo:hi], _expert(w13, e), _expert(w2, e))
        if h is None:
            h = np.zeros((nK, G_e.shape[1]), dtype=F64)
        h[lo:hi] = G_e
        y_perm[lo:hi] = Y_e
    return h, y_perm


def combine(y_perm, w_top, inv_perm):
    """Steps 10-11: y[i] = sum_k w_top[i, k] * Y[inv_perm[i*K + k]]."""
    w_top = _f64(w_top)
    n, K = w_top.shape
    y_perm = _f64(y_perm)
    y = np.zeros((n, y_perm.shape[1]), dtype=F64)
    inv = np.asarray(inv_perm).reshape(n, K)
    for k in range(K):
        y += w_top[:, k:k + 1] * y_perm[inv[:, k]]
    return y


# --------------------------------------------------------------------------
# The whole layer
# --------------------------------------------------------------------------

def moe_forward(x, w_gate, bias, w13, w2, K, norm_topk_prob, forced=None):
    """Algorithm 2 end to end.  `w13`/`w2` are (E, ...) arrays or callables
    e -> slice.  `forced` = (token_ids, e_top_rows) imposes the expert choice
    (and slot order) of the listed tokens -- used for near-tie tokens, whose
    choice is decided by rounding; their weights are still the oracle's p.

    Returns a dict with every intermediate: logits, p, e_top, w_top, counts,
    offsets, perm, inv_perm, h, y_perm, y.
    """
    x = _f64(x)
    logits = router_logits(x, w_gate, bias)
    E = logits.shape[1]
    e_top, w_top = topk(logits, K, norm_topk_prob)
    if forced is not None:
        ids, rows = forced
        ids = np.asarray(ids, dtype=np.int64)
        if ids.size:
            e_top[ids] = np.asarray(rows, dtype=np.int64)
            w_top[ids] = weights_for(logits[ids], e_top[ids], norm_topk_prob)
    counts, offsets, perm, inv_perm = dispatch_layout(e_top, E)
    x_perm = permute(x, perm, K)
    h, y_perm = grouped_swiglu(x_perm, offsets, w13, w2)
    y = combine(y_perm, w_top, inv_perm)
    return dict(logits=logits, p=softmax(logits), e_top=e_top, w_top=w_top,
                counts=counts, offsets=offsets, perm=perm, inv_perm=inv_perm,
                h=h, y_perm=y_perm, y=y)


def count_cv(counts):
    """Imbalance of the per-expert hit counts: CV = sigma_e(n_e) / mu_e(n_e)
    (population standard deviation), as quantified in §1.2."""
    c = np.asarray(counts, dtype=F64)
    return float(np.std(c) / np.mean(c))
