"""The CPU oracle against its pins (no GPU)."""
import numpy as np
import pytest

from oracle import brute
from oracle import moe_oracle as O
from tests import oracle_pins as P
from workloads import TINY, SKEW, synth


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(O)


@pytest.mark.parametrize("kw", [
    dict(n=20, H=12, I=6, E=5, K=2),
    dict(n=16, H=9, I=5, E=7, K=3, bias=True, cold=2),   # two experts never chosen
    dict(n=8, H=6, I=3, E=4, K=4),                       # K = E
    dict(n=1, H=4, I=2, E=3, K=1),                       # one token
])
def test_brute_force_shapes(kw):
    P.pin_brute_force(O, seed=11, **kw)


def test_brute_force_on_tiny_workload():
    """The tiny workload's own inputs (CPU draws), 12 tokens brute-forced."""
    cfg = TINY
    x = synth.to_f64_numpy(synth.make_x(cfg, "cpu"))
    L = synth.make_layer(cfg, "cpu")
    wg, w13, w2 = (synth.to_f64_numpy(L[k]) for k in ("w_gate", "w13", "w2"))
    r = O.moe_forward(x, wg, None, w13, w2, cfg.K, cfg.norm_topk_prob)
    toks = list(range(0, cfg.n, cfg.n // 12))[:12]
    be, bw, by = brute.moe_forward_brute(x, wg, None, w13, w2, cfg.K, cfg.norm_topk_prob, toks)
    assert r["e_top"][toks].tolist() == be
    assert np.allclose(r["w_top"][toks], bw, rtol=1e-12)
    assert np.allclose(r["y"][toks], by, rtol=1e-11, atol=1e-12)


def test_empty_experts_skipped():
    x, wg, b, w13, w2 = P.small_case(2, n=40, H=8, I=4, E=6, K=2, bias=True, cold=3)
    r = O.moe_forward(x, wg, b, w13, w2, 2, False)
    assert list(r["counts"][:3]) == [0, 0, 0]
    assert r["offsets"][0] == r["offsets"][3] == 0
    # garbage weights of never-chosen experts cannot leak into y
    w13b = w13.copy()
    w13b[:3] = np.nan
    r2 = O.moe_forward(x, wg, b, w13b, w2, 2, False)
    assert np.array_equal(r["y"], r2["y"])


def test_near_tie_detection():
    logits = np.array([
        [3.0, 2.0, 1.0, 0.0],
        [3.0, 2.0, 2.0 - 5e-7, 0.0],      # boundary tie for K=2
        [3.0, 3.0 - 5e-7, 1.0, 0.0],      # in-set order tie
        [3.0, 2.0, 1.0, 1.0],             # tie below the K+1-th: harmless
        [3.0, -np.inf, -np.inf, -np.inf],  # equal infinite logits at the boundary
    ])
    assert O.near_tie_tokens(logits, 2).tolist() == [False, True, True, False, True]
    assert O.near_tie_tokens(logits, 2, gap=2.0).tolist() == [True, True, True, True, True]


def test_forced_choice():
    x, wg, b, w13, w2 = P.small_case(9, n=12, H=8, I=4, E=5, K=2)
    r = O.moe_forward(x, wg, b, w13, w2, 2, True)
    same = O.moe_forward(x, wg, b, w13, w2, 2, True, forced=([3, 7], r["e_top"][[3, 7]]))
    assert np.array_equal(same["y"], r["y"])
    alt = r["e_top"][[3]][:, ::-1].copy()         # same set, other slot order
    r2 = O.moe_forward(x, wg, b, w13, w2, 2, True, forced=([3], alt))
    assert r2["e_top"][3].tolist() == alt[0].tolist()
    assert np.allclose(r2["y"], r["y"], rtol=1e-13, atol=1e-14)   # y does not depend on slot order
    other = np.array([[r["e_top"][3][0], [e for e in range(5) if e not in r["e_top"][3]][0]]])
    r3 = O.moe_forward(x, wg, b, w13, w2, 2, True, forced=([3], other))
    assert not np.allclose(r3["y"][3], r["y"][3])
    assert np.allclose(np.delete(r3["y"], 3, 0), np.delete(r["y"], 3, 0))


def test_streamed_weights_match_arrays():
    x, wg, b, w13, w2 = P.small_case(4, n=25, H=8, I=4, E=6, K=3)
    r = O.moe_forward(x, wg, b, w13, w2, 3, False)
    r2 = O.moe_forward(x, wg, b, lambda e: w13[e], lambda e: w2[e], 3, False)
    assert np.array_equal(r["y"], r2["y"])


def test_skew_bias_shape():
    b = synth.skew_bias(SKEW).numpy()
    assert b.shape == (SKEW.E,)
    assert int(np.isneginf(b).sum()) == 4
    fin = b[np.isfinite(b)]
    assert fin.max() == 0.0                      # rank 1 gets ln(1) = 0
    assert np.all(fin <= 0)


def test_count_cv():
    assert O.count_cv([2, 2, 2, 2]) == 0.0
    assert abs(O.count_cv([0, 0, 0, 4]) - np.sqrt(3.0)) < 1e-15
