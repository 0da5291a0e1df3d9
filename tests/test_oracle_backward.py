"""Pins of the backward oracle (oracle/moe_backward.py), CPU only.

The backward is pinned to the forward oracle, which is pinned on its own
(tests/oracle_pins.py): for L = <dy, y>, every gradient the backward returns
must match central finite differences of the forward in float64, with the
expert choice held at the unperturbed one (the choice is a step function;
the backward differentiates with it fixed).  Plus the invariants the
mathematics fixes: a softmax gradient sums to zero per token; with one expert
the routing weight is 1 and the router receives no gradient.  Finally,
plausible mistakes planted in a copy of the backward must each fail a pin."""
import importlib.util

import numpy as np
import pytest

from oracle import moe_oracle as F
from oracle import moe_backward as _B

EPS = 1e-6


def _problem(seed, n=6, H=8, I=4, E=4, K=2, bias=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, H))
    w_gate = rng.standard_normal((H, E)) * 0.5
    b = rng.standard_normal(E) * 0.3 if bias else None
    w13 = rng.standard_normal((E, H, 2 * I)) / np.sqrt(H)
    w2 = rng.standard_normal((E, I, H)) / np.sqrt(I)
    dy = rng.standard_normal((n, H))
    return x, w_gate, b, w13, w2, dy


def _loss(x, w_gate, b, w13, w2, K, norm, dy, forced):
    return float(np.sum(dy * F.moe_forward(x, w_gate, b, w13, w2, K, norm, forced=forced)["y"]))


def _check_fd(B, seed, K, norm, bias, coords=6):
    x, w_gate, b, w13, w2, dy = _problem(seed, K=K, bias=bias)
    g = B.moe_backward(x, w_gate, b, w13, w2, K, norm, dy)
    forced = (np.arange(x.shape[0]), g["e_top"])
    rng = np.random.default_rng(seed + 100)
    params = dict(x=x, w_gate=w_gate, w13=w13, w2=w2)
    grads = dict(x=g["dx"], w_gate=g["dw_gate"], w13=g["dw13"], w2=g["dw2"])
    if bias:
        params["b"] = b
        grads["b"] = g["dbias"]
    worst = 0.0
    for name, arr in params.items():
        for _ in range(coords):
            idx = tuple(rng.integers(0, s) for s in arr.shape)
            args = dict(x=x, w_gate=w_gate, b=b, w13=w13, w2=w2)
            plus = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in args.items()}
            minus = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in args.items()}
            plus[name][idx] += EPS
            minus[name][idx] -= EPS
            fd = (_loss(**plus, K=K, norm=norm, dy=dy, forced=forced) -
                  _loss(**minus, K=K, norm=norm, dy=dy, forced=forced)) / (2 * EPS)
            err = abs(fd - grads[name][idx]) / (1.0 + abs(fd))
            worst = max(worst, err)
    return worst


@pytest.mark.parametrize("seed,K,norm,bias", [(1, 2, True, True), (2, 2, False, True),
                                              (3, 3, True, False), (4, 1, False, False)])
def test_backward_matches_finite_differences(seed, K, norm, bias):
    assert _check_fd(_B, seed, K, norm, bias) < 1e-6


def test_softmax_gradient_sums_to_zero_per_token():
    x, w_gate, b, w13, w2, dy = _problem(5)
    g = _B.moe_backward(x, w_gate, b, w13, w2, 2, True, dy)
    assert np.max(np.abs(g["dlogits"].sum(axis=1))) < 1e-12
    assert np.allclose(g["dbias"], g["dlogits"].sum(axis=0))


def test_one_expert_router_gets_no_gradient():
    """E = 1, K = 1: the weight is softmax of one logit = 1 for every input,
    so the router's gradients vanish and dx is the dense SwiGLU MLP's."""
    x, w_gate, b, w13, w2, dy = _problem(6, E=1, K=1, bias=False)
    g = _B.moe_backward(x, w_gate, None, w13, w2, 1, False, dy)
    assert np.max(np.abs(g["dlogits"])) == 0.0
    assert np.max(np.abs(g["dw_gate"])) == 0.0
    assert np.allclose(g["dx"], g["dx_experts"])


def test_single_renormalised_slot_gives_no_router_gradient():
    """K = 1 with renormalisation: the weight w = p_e / p_e is 1 whatever the
    logits, so the router gets no gradient although E > 1."""
    x, w_gate, b, w13, w2, dy = _problem(8, E=4, K=1)
    g = _B.moe_backward(x, w_gate, b, w13, w2, 1, True, dy)
    assert np.max(np.abs(g["dlogits"])) == 0.0
    assert np.max(np.abs(g["dw_gate"])) == 0.0 and np.max(np.abs(g["dbias"])) == 0.0
    assert np.max(np.abs(g["dw"])) > 0.0  # the slot weight's own gradient is not zero


def test_pairs_of_one_token_sum_in_dx():
    """The permute backward adds the K slot rows of a token: with K copies of
    the same expert impossible, check dx_experts against a per-pair sum."""
    x, w_gate, b, w13, w2, dy = _problem(7, K=3)
    g = _B.moe_backward(x, w_gate, b, w13, w2, 3, True, dy)
    inv = g["inv_perm"].reshape(x.shape[0], 3)
    manual = sum(g["dx_perm"][inv[:, k]] for k in range(3))
    assert np.allclose(manual, g["dx_experts"], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- mutations
def _fresh():
    spec = importlib.util.spec_from_file_location("oracle.moe_backward_copy", _B.__file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _sigmoid_only(M):  # d silu / dG written as sigmoid(G) alone
    orig = M.expert_backward

    def eb(X_e, W13_e, W2_e, dY_e):
        out = orig(X_e, W13_e, W2_e, dY_e)
        I = W13_e.shape[1] // 2
        gu = X_e @ W13_e
        G, U = gu[:, :I], gu[:, I:]
        s = 1 / (1 + np.exp(-G))
        dG = out["dh"] * U * s
        out["dGU"] = np.concatenate([dG, out["dU"]], axis=1)
        out["dX"] = out["dGU"] @ W13_e.T
        out["dW13"] = X_e.T @ out["dGU"]
        return out
    M.expert_backward = eb


def _no_renorm_term(M):  # renormalisation ignored in the router backward
    orig = M.router_backward
    M.router_backward = lambda x, wg, lg, et, wt, dw, norm: orig(x, wg, lg, et, wt, dw, False)


def _unweighted_dY(M):  # combine backward without the routing weight
    orig = M.combine_backward

    def cb(dy, y_perm, w_top, inv_perm):
        dY, dw = orig(dy, y_perm, np.ones_like(np.asarray(w_top, dtype=float)), inv_perm)
        return dY, dw
    M.combine_backward = cb


def _halved_dw2(M):  # a factor dropped from dW2
    orig = M.expert_backward

    def eb(X_e, W13_e, W2_e, dY_e):
        out = orig(X_e, W13_e, W2_e, dY_e)
        out["dW2"] = out["dW2"] * 0.5
        return out
    M.expert_backward = eb


@pytest.mark.parametrize("mutate", [_sigmoid_only, _no_renorm_term, _unweighted_dY,
                                    _halved_dw2], ids=lambda f: f.__name__)
def test_planted_mistakes_fail_a_pin(mutate):
    M = _fresh()
    mutate(M)
    worst = max(_check_fd(M, seed, K, norm, bias)
                for seed, K, norm, bias in [(1, 2, True, True), (3, 3, True, False)])
    assert worst > 1e-4, worst
