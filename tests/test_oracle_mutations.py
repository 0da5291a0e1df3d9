"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them (CPU only; the real oracle is never modified)."""
import importlib.util
import types

import numpy as np
import pytest

from oracle import moe_oracle as _O
from tests import oracle_pins as P


def _fresh_oracle():
    spec = importlib.util.spec_from_file_location("oracle_copy", _O.__file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _swap_gate_up(M):
    def expert_up(X_e, W13_e):
        I = W13_e.shape[1] // 2
        gu = X_e @ W13_e
        up, gate = gu[:, :I], gu[:, I:]
        return gate / (1.0 + np.exp(-gate)) * up
    M.expert_up = expert_up


def _silu_sign(M):
    def expert_up(X_e, W13_e):
        I = W13_e.shape[1] // 2
        gu = X_e @ W13_e
        gate, up = gu[:, :I], gu[:, I:]
        return gate / (1.0 + np.exp(gate)) * up
    M.expert_up = expert_up


def _drop_renorm(M):
    orig = M.topk
    M.topk = lambda logits, K, norm: orig(logits, K, False)


def _ascending_topk(M):
    def topk(logits, K, norm):
        order = np.argsort(logits, axis=1, kind="stable")[:, :K]
        w = np.take_along_axis(M.softmax(logits), order, 1)
        if norm:
            w = w / w.sum(1, keepdims=True)
        return order, w
    M.topk = topk


def _ties_to_higher_index(M):
    def topk(logits, K, norm):
        E = logits.shape[1]
        order = (E - 1 - np.argsort(-logits[:, ::-1], axis=1, kind="stable"))[:, :K]
        w = np.take_along_axis(M.softmax(logits), order, 1)
        if norm:
            w = w / w.sum(1, keepdims=True)
        return order, w
    M.topk = topk


def _slot_major_flat(M):
    orig = M.dispatch_layout

    def dispatch_layout(e_top, E):
        e_top = np.asarray(e_top)
        counts, offsets, perm, inv = orig(e_top.T.copy(), E)   # f = k*n + t
        return counts, offsets, perm, inv
    M.dispatch_layout = dispatch_layout


def _unstable_sort(M):
    orig = M.dispatch_layout

    def dispatch_layout(e_top, E):
        counts, offsets, perm, inv = orig(e_top, E)
        perm = perm.copy()
        for e in range(E):                      # reverse each expert's run
            perm[offsets[e]:offsets[e + 1]] = perm[offsets[e]:offsets[e + 1]][::-1]
        inv = np.empty_like(perm)
        inv[perm] = np.arange(perm.size)
        return counts, offsets, perm, inv
    M.dispatch_layout = dispatch_layout


def _combine_with_perm(M):
    def combine(y_perm, w_top, inv_perm):
        n, K = w_top.shape
        inv = np.empty_like(np.asarray(inv_perm))
        inv[np.asarray(inv_perm)] = np.arange(inv.size)      # uses perm, not inv_perm
        y = np.zeros((n, y_perm.shape[1]))
        inv = inv.reshape(n, K)
        for k in range(K):
            y += w_top[:, k:k + 1] * y_perm[inv[:, k]]
        return y
    M.combine = combine


def _ignore_bias(M):
    orig = M.router_logits
    M.router_logits = lambda x, w_gate, bias=None: orig(x, w_gate, None)


def _softmax_wrong_axis(M):
    def softmax(logits):
        logits = np.asarray(logits, dtype=np.float64)
        z = np.exp(logits - logits.max(0, keepdims=True))
        return z / z.sum(0, keepdims=True)
    M.softmax = softmax


def _gather_by_flat_not_token(M):
    M.permute = lambda x, perm, K: np.asarray(x, dtype=np.float64)[np.asarray(perm) % x.shape[0]]


def _w2_rows_reversed(M):
    M.expert_down = lambda G_e, W2_e: G_e @ W2_e[::-1]       # wrong row index into W2


MUTATIONS = [_swap_gate_up, _silu_sign, _drop_renorm, _ascending_topk, _ties_to_higher_index,
             _slot_major_flat, _unstable_sort, _combine_with_perm, _ignore_bias,
             _softmax_wrong_axis, _gather_by_flat_not_token, _w2_rows_reversed]


@pytest.mark.parametrize("mutate", MUTATIONS, ids=lambda f: f.__name__.strip("_"))
def test_pins_catch_mutation(mutate):
    M = _fresh_oracle()
    mutate(M)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(M)
        except Exception as exc:   # AssertionError, or a crash the mistake causes
            caught.append((pin.__name__, type(exc).__name__))
    assert caught, f"no pin caught {mutate.__name__}"


def test_unmutated_copy_passes():
    M = _fresh_oracle()
    for pin in P.ALL_PINS:
        pin(M)
    assert isinstance(M, types.ModuleType)
