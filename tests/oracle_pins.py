"""Pins of the fp64 oracle: checks against things other than the oracle itself.

Each `pin_*` function runs one check against the module object `O` it is
given and raises AssertionError on failure, so the same pins can be pointed
at a deliberately broken copy of the oracle (tests/test_oracle_mutations.py)
to show that they catch plausible mistakes.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

from oracle import brute

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def small_case(seed, n=20, H=12, I=6, E=5, K=2, bias=False, cold=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, H))
    wg = rng.standard_normal((H, E)) * 0.3
    w13 = rng.standard_normal((E, H, 2 * I)) / math.sqrt(H)
    w2 = rng.standard_normal((E, I, H)) / math.sqrt(I)
    b = None
    if bias:
        b = rng.standard_normal(E) * 0.5
        if cold:
            b[:cold] = -np.inf
    return x, wg, b, w13, w2


def pin_align_block_size_example(O):
    """The worked `moe_align_block_size` example (E=4, BLOCK_SIZE_M=4)."""
    g = json.load(open(os.path.join(GOLDEN, "align_block_size_example.json")))
    ids = np.array(g["topk_ids_as_printed"]) - g["id_shift"]
    counts, offsets, perm, inv = O.dispatch_layout(ids, g["E"])
    sorted_ids, expert_ids, total = O.padded_block_layout(
        counts, offsets, perm, g["block_size_m"], "PAD")
    assert [int(v) if v != "PAD" else v for v in sorted_ids] == g["sorted_token_ids_as_printed"]
    assert expert_ids == g["expert_ids_as_printed"]
    assert total == g["num_tokens_post_padded"]
    assert list(counts) == [3, 3, 3, 3]
    assert list(offsets) == [0, 3, 6, 9, 12]


def pin_swiglu_hand(O):
    """A SwiGLU expert computed by hand, through the whole layer (E=1, K=1)."""
    g = json.load(open(os.path.join(GOLDEN, "silu_swiglu_hand.json")))
    x = np.array(g["x"])
    w13 = np.array(g["w13"])
    w2 = np.array(g["w2"])
    wg = np.zeros((x.shape[1], 1))
    r = O.moe_forward(x, wg, None, w13, w2, K=1, norm_topk_prob=False)
    assert np.allclose(r["h"], g["h"], rtol=1e-15, atol=0)
    assert np.allclose(r["y"], g["y_single_expert"], rtol=1e-15, atol=0)


def pin_softmax_closed_form(O):
    p = O.softmax(np.array([[0.0, math.log(3.0)], [5.0, -np.inf]]))
    assert np.allclose(p, [[0.25, 0.75], [1.0, 0.0]], rtol=1e-15, atol=1e-300)
    # shift invariance and a large-logit row that would overflow an unshifted exp
    p2 = O.softmax(np.array([[1000.0, 1000.0 + math.log(3.0)]]))
    assert np.allclose(p2, [[0.25, 0.75]], rtol=1e-14)


def pin_topk_order_and_ties(O):
    """Descending logit order; equal logits go to the lower expert index."""
    logits = np.array([[1.0, 3.0, 3.0, 2.0], [0.5, -1.0, 0.5, 0.5]])
    e, w = O.topk(logits, 2, False)
    assert e.tolist() == [[1, 2], [0, 2]]
    p = np.exp(logits) / np.exp(logits).sum(1, keepdims=True)
    assert np.allclose(w, [[p[0, 1], p[0, 2]], [p[1, 0], p[1, 2]]], rtol=1e-15)
    e3, w3 = O.topk(logits, 3, True)
    assert e3.tolist() == [[1, 2, 3], [0, 2, 3]]
    assert np.allclose(w3.sum(1), 1.0, rtol=1e-15)


def pin_brute_force(O, seed=0, **kw):
    """Oracle == pure-Python per-token loop on a small random case."""
    for norm in (False, True):
        x, wg, b, w13, w2 = small_case(seed, **kw)
        K = kw.get("K", 2)
        r = O.moe_forward(x, wg, b, w13, w2, K, norm)
        be, bw, by = brute.moe_forward_brute(x, wg, b, w13, w2, K, norm)
        assert r["e_top"].tolist() == be
        assert np.allclose(r["w_top"], np.array(bw), rtol=1e-12, atol=0)
        by = np.array(by)
        err = np.linalg.norm(r["y"] - by) / np.linalg.norm(by)
        assert err < 1e-12, err


def pin_layout_invariants(O, seed=3, n=300, E=16, K=4):
    """counts sum to n*K; perm is a permutation; inv_perm inverts it; every
    expert segment holds only that expert's pairs, in ascending flat index;
    and the layout agrees with a direct per-expert scan over the pairs."""
    rng = np.random.default_rng(seed)
    e_top = np.stack([rng.permutation(E)[:K] for _ in range(n)])
    e_top[:40] = np.arange(K)            # a hot set of experts
    counts, offsets, perm, inv = O.dispatch_layout(e_top, E)
    flat = e_top.reshape(-1)
    assert counts.sum() == n * K
    assert offsets[0] == 0 and offsets[-1] == n * K
    assert sorted(perm.tolist()) == list(range(n * K))
    assert np.array_equal(inv[perm], np.arange(n * K))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)
        assert seg.tolist() == [f for f in range(n * K) if flat[f] == e]


def pin_router_invariants(O, seed=4):
    x, wg, b, *_ = small_case(seed, n=200, H=16, E=12, bias=True, cold=3)
    logits = O.router_logits(x, wg, b)
    direct = np.array([[sum(x[t, h] * wg[h, e] for h in range(16)) + b[e]
                        for e in range(12)] for t in range(5)])
    assert np.allclose(logits[:5], direct, rtol=1e-13, atol=1e-13)
    e_n, w_n = O.topk(logits, 4, True)
    e_u, w_u = O.topk(logits, 4, False)
    assert np.array_equal(e_n, e_u)
    assert np.allclose(w_n.sum(1), 1.0, atol=1e-12)
    assert np.all(w_u.sum(1) <= 1.0 + 1e-12)
    assert np.all(np.diff(w_u, axis=1) <= 0)
    for row in e_n:
        assert len(set(row.tolist())) == 4 and all(3 <= v < 12 for v in row)  # cold never chosen


def pin_e1_k1_dense(O, seed=5):
    """E=1, K=1: the layer reduces to a dense SwiGLU MLP with weight 1."""
    x, wg, _, w13, w2 = small_case(seed, n=17, H=10, I=7, E=1)
    r = O.moe_forward(x, wg, None, w13, w2, K=1, norm_topk_prob=False)
    W1, W3 = w13[0][:, :7], w13[0][:, 7:]
    a = x @ W1
    dense = (a * (0.5 * (1.0 + np.tanh(0.5 * a)))) * (x @ W3) @ w2[0]  # sigmoid via tanh
    assert np.allclose(r["w_top"], 1.0, rtol=0, atol=0)
    assert np.allclose(r["y"], dense, rtol=1e-12, atol=1e-13)


def pin_all_experts(O, seed=6):
    """K = E: every expert is chosen, y = sum_e p_e * SwiGLU_e(x) densely."""
    x, wg, _, w13, w2 = small_case(seed, n=9, H=8, I=4, E=3, K=3)
    r = O.moe_forward(x, wg, None, w13, w2, K=3, norm_topk_prob=False)
    logits = x @ wg
    p = np.exp(logits) / np.exp(logits).sum(1, keepdims=True)
    y = np.zeros_like(x)
    for e in range(3):
        g = x @ w13[e][:, :4]
        u = x @ w13[e][:, 4:]
        y += p[:, e:e + 1] * (((g * (0.5 * (1.0 + np.tanh(0.5 * g)))) * u) @ w2[e])
    assert np.allclose(r["y"], y, rtol=1e-12, atol=1e-13)


def pin_token_equivariance(O, seed=7):
    x, wg, b, w13, w2 = small_case(seed, n=30, H=8, I=4, E=6, K=3, bias=True)
    r = O.moe_forward(x, wg, b, w13, w2, 3, True)
    sh = np.random.default_rng(seed).permutation(30)
    r2 = O.moe_forward(x[sh], wg, b, w13, w2, 3, True)
    assert np.allclose(r2["y"], r["y"][sh], rtol=1e-13, atol=1e-14)


ALL_PINS = [
    pin_align_block_size_example,
    pin_swiglu_hand,
    pin_softmax_closed_form,
    pin_topk_order_and_ties,
    pin_brute_force,
    pin_layout_invariants,
    pin_router_invariants,
    pin_e1_k1_dense,
    pin_all_experts,
    pin_token_equivariance,
]
