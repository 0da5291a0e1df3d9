"""GPU parity: every step of the layer against the fp64 oracle, through the
C ABI.  Sizes the oracle finishes in seconds are compared element by element;
the full workloads are compared on every token for routing/layout and on
sampled tokens for the expert outputs."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from tests.gpu_helpers import (Run, TOL, rel_fro, valid_near_tie_choice, f64, tie_margin,
                               logit_error_within_margin)
from workloads import TINY, OLMOE, SKEW, DSV3
from workloads.configs import MoEConfig

pytestmark = pytest.mark.gpu

# small shapes that still span several tiles and a ragged tail
SMALL = [
    TINY,
    OLMOE.with_(name="olmoe_n512", n=512),
    MoEConfig("ragged_bf16", n=333, H=192, I=256, E=16, K=4, dtype="bf16",
              norm_topk_prob=True, seed=21),
    MoEConfig("ragged_skew_bf16", n=300, H=256, I=128, E=12, K=3, dtype="bf16",
              norm_topk_prob=False, seed=22, skew=True),
    MoEConfig("one_expert_bf16", n=130, H=128, I=128, E=1, K=1, dtype="bf16",
              norm_topk_prob=False, seed=23),
    MoEConfig("k_equals_e_f32", n=50, H=64, I=32, E=4, K=4, dtype="f32",
              norm_topk_prob=True, seed=24),
    MoEConfig("one_token_bf16", n=1, H=128, I=128, E=8, K=2, dtype="bf16",
              norm_topk_prob=True, seed=25),
    # tensor-core router path (E % 64 == 0): ragged tail tile, bias with -inf experts
    MoEConfig("ragged_e64_skew_bf16", n=333, H=256, I=128, E=64, K=6, dtype="bf16",
              norm_topk_prob=True, seed=26, skew=True),
    MoEConfig("e128_k3_bf16", n=700, H=320, I=256, E=128, K=3, dtype="bf16",
              norm_topk_prob=False, seed=27),
]
FULL = [OLMOE, SKEW, DSV3]


def check_router(run, rows=None):
    cfg = run.cfg
    lo = run.oracle_logits()
    lg = run.np("logits")
    near = O.near_tie_tokens(lo, cfg.K)
    gi = run.np("topk_idx")
    gw = run.np("topk_w")
    oe, ow = O.topk(lo, cfg.K, cfg.norm_topk_prob)
    ok = ~near
    assert np.array_equal(gi[ok], oe[ok]), "TopK indices differ on non-near-tie tokens"
    for t in np.where(near)[0]:
        assert valid_near_tie_choice(lo[t], gi[t], cfg.K), f"token {t}: invalid near-tie choice"
    # float32 logits: inside half the near-tie rescoring margin for every
    # token, so every token the kernel did not rescore is ordered right
    ok_m, ratio, err = logit_error_within_margin(lg, lo, tie_margin(cfg))
    print(f"{cfg.name}: max logit error {err:.3e}, worst error / half-margin {ratio:.3f}")
    assert ok_m, (ratio, err)
    # softmax weights move by at most ~2x the largest logit error (relative),
    # plus float32 rounding of exp and the divisions
    rel = np.abs(gw[ok] - ow[ok]) / np.maximum(np.abs(ow[ok]), 1e-30)
    assert rel.max(initial=0) <= 2.0 * err + 2e-6, (rel.max(), err)
    return err, int(near.sum())


def check_layout(run):
    cfg = run.cfg
    gi = run.np("topk_idx")
    counts, offsets, perm, inv = O.dispatch_layout(gi, cfg.E)
    assert np.array_equal(run.np("counts"), counts)
    assert np.array_equal(run.np("offsets"), offsets)
    assert np.array_equal(run.np("perm"), perm)
    assert np.array_equal(run.np("inv_perm"), inv)


def run_permute(run):
    """x_perm from an explicit moe_permute call on the layer's own layout, into
    a fresh buffer."""
    import top_routing_dispatch_gb300 as M
    xp = torch.empty((run.cfg.nK, run.cfg.H), dtype=run.x.dtype, device=run.dev)
    st = torch.zeros(1, dtype=torch.int32, device=run.dev)
    M.moe_permute(run.desc, run.x, run.view("perm"), xp, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return xp


def check_permute(run, sample_rows=None):
    """x_perm against the oracle's gather, exactly (bf16/f32 -> f64 is exact)."""
    perm = run.np("perm")
    xp = run_permute(run)
    if sample_rows is None:
        assert np.array_equal(f64(xp), O.permute(f64(run.x), perm, run.cfg.K))
        return
    r = np.asarray(sample_rows)
    got = f64(xp[torch.as_tensor(r, device=xp.device)])
    ref = O.permute(f64(run.x), perm[r], run.cfg.K)
    assert np.array_equal(got, ref)


def check_permute_scatter(run, sample_rows=None):
    """The scatter form (x read once, written to the K rows inv_perm names)
    against the oracle's gather, exactly; the destination starts as all-ones
    bytes so a row the kernel misses cannot pass."""
    import top_routing_dispatch_gb300 as M
    xp = torch.full((run.cfg.nK, run.cfg.H), -1, dtype=torch.int16,
                    device=run.dev).view(run.x.dtype) if run.x.dtype == torch.bfloat16 else \
        torch.full((run.cfg.nK, run.cfg.H), float("nan"), dtype=run.x.dtype, device=run.dev)
    st = torch.zeros(1, dtype=torch.int32, device=run.dev)
    M.moe_permute_scatter(run.desc, run.x, run.view("inv_perm"), xp, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    perm = run.np("perm")
    if sample_rows is None:
        assert np.array_equal(f64(xp), O.permute(f64(run.x), perm, run.cfg.K))
        return
    r = np.asarray(sample_rows)
    got = f64(xp[torch.as_tensor(r, device=xp.device)])
    assert np.array_equal(got, O.permute(f64(run.x), perm[r], run.cfg.K))
    # every row, against the gather form (itself checked against the oracle)
    assert torch.equal(xp.view(torch.int16) if xp.dtype == torch.bfloat16 else xp,
                       run_permute(run).view(torch.int16) if xp.dtype == torch.bfloat16
                       else run_permute(run))


def check_experts(run, sample_rows=None):
    """GPU h and the GEMM2 output against the oracle's SwiGLU: GEMM1 on the
    oracle's gather of x (Algorithm 2 step 7), GEMM2 on the GPU's (rounded) h.
    bf16 layers: the workspace holds y_slot[perm[r]] = w[perm[r]] * Y[r]
    (moe_expert_gemm2_weighted); float32 layers: y_perm[r] = Y[r]."""
    cfg = run.cfg
    off = run.np("offsets")
    perm = run.np("perm")
    tw = run.np("topk_w").reshape(-1)
    h = run.view("h")
    yp = run.view("y_perm")
    nK = cfg.nK
    rows = np.arange(nK) if sample_rows is None else np.asarray(sorted(set(sample_rows)))
    experts = np.searchsorted(off, rows, side="right") - 1
    x64 = f64(run.x)
    weighted = cfg.dtype == "bf16"
    hs, ys, ho, yo = [], [], [], []
    for e in np.unique(experts):
        r = rows[experts == e]
        ri = torch.as_tensor(r, device=h.device)
        ho.append(O.expert_up(O.permute(x64, perm[r], cfg.K), run.w13_get(int(e))))
        ye = O.expert_down(f64(h[ri]), run.w2_get(int(e)))
        if weighted:
            f = perm[r]
            yo.append(ye * tw[f][:, None])
            ys.append(f64(yp[torch.as_tensor(f, device=yp.device)]))
        else:
            yo.append(ye)
            ys.append(f64(yp[ri]))
        hs.append(f64(h[ri]))
    tol = TOL[cfg.dtype]
    eh = rel_fro(np.concatenate(hs), np.concatenate(ho))
    ey = rel_fro(np.concatenate(ys), np.concatenate(yo))
    assert eh <= tol, f"h error {eh:.3e}"
    assert ey <= tol, f"y_perm error {ey:.3e}"
    return eh, ey


def check_unweighted_gemm2_and_combine(run, sample_rows=None):
    """bf16: the unweighted pair moe_expert_gemm2 + moe_combine on the same h,
    against the oracle and against the forward's y."""
    import top_routing_dispatch_gb300 as M
    cfg = run.cfg
    if cfg.dtype != "bf16":
        return
    yp = torch.empty((cfg.nK, cfg.H), dtype=run.x.dtype, device=run.dev)
    y = torch.empty_like(run.x)
    st = torch.zeros(1, dtype=torch.int32, device=run.dev)
    M.moe_expert_gemm2(run.desc, run.view("h"), run.L["w2"], run.view("offsets"), yp,
                       status_word=st)
    M.moe_combine(run.desc, yp, run.view("topk_w"), run.view("inv_perm"), y, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    off = run.np("offsets")
    h = run.view("h")
    rows = np.arange(cfg.nK) if sample_rows is None else np.asarray(sorted(set(sample_rows)))
    experts = np.searchsorted(off, rows, side="right") - 1
    ys, yo = [], []
    for e in np.unique(experts):
        r = rows[experts == e]
        ri = torch.as_tensor(r, device=h.device)
        yo.append(O.expert_down(f64(h[ri]), run.w2_get(int(e))))
        ys.append(f64(yp[ri]))
    assert rel_fro(np.concatenate(ys), np.concatenate(yo)) <= TOL[cfg.dtype]
    # the same layer output up to the two bf16 roundings of y_perm vs y_slot
    assert rel_fro(f64(y), f64(run.y)) <= 8e-3


def check_gather_fusion(run):
    """bf16: GEMM1 with the gather fused into its A loads gives the same bits
    as moe_permute followed by the unfused GEMM1 (each h row depends on its
    own A row only, and both read the same values)."""
    import top_routing_dispatch_gb300 as M
    cfg = run.cfg
    if cfg.dtype != "bf16" or cfg.I % 128 or cfg.H % 64:
        return
    xp = run_permute(run)
    h1 = torch.empty((cfg.nK, cfg.I), dtype=run.x.dtype, device=run.dev)
    h2 = torch.empty_like(h1)
    st = torch.zeros(1, dtype=torch.int32, device=run.dev)
    off = run.view("offsets")
    M.moe_expert_gemm1_swiglu(run.desc, xp, run.L["w13"], off, h1, status_word=st)
    M.moe_expert_gemm1_swiglu_gather(run.desc, run.x, run.view("perm"), run.L["w13"], off, h2,
                                     status_word=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(h1.view(torch.int16), h2.view(torch.int16))
    # and both equal the h of the forward
    assert torch.equal(h2.view(torch.int16), run.view("h").view(torch.int16))


def check_combine(run):
    cfg = run.cfg
    if cfg.dtype == "bf16":   # y[t] = sum of the token's K weighted slot rows
        ys = run.np("y_perm").reshape(cfg.n, cfg.K, cfg.H)
        yo = ys.sum(axis=1)
    else:
        yo = O.combine(run.np("y_perm"), run.np("topk_w"), run.np("inv_perm"))
    err = rel_fro(f64(run.y), yo)
    assert err <= (4e-3 if cfg.dtype == "bf16" else 1e-6), err


def check_layer(run, rows=None):
    r = run.oracle_layer(rows)
    y = f64(run.y) if rows is None else f64(run.y[torch.as_tensor(rows, device=run.y.device)])
    err = rel_fro(y, r["y"])
    assert err <= TOL[run.cfg.dtype], f"layer error {err:.3e}"
    gi = run.np("topk_idx") if rows is None else run.np("topk_idx")[np.asarray(rows)]
    ok = ~r["near"]
    assert np.array_equal(gi[ok], r["e_top"][ok])
    return err


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_small_all_steps(cfg):
    run = Run(cfg)
    assert run.status == 0
    check_router(run)
    check_layout(run)
    check_permute(run)
    check_permute_scatter(run)
    check_experts(run)
    check_gather_fusion(run)
    check_unweighted_gemm2_and_combine(run)
    check_combine(run)
    check_layer(run)


@pytest.mark.parametrize("cfg", FULL, ids=lambda c: c.name)
def test_full_size(cfg):
    run = Run(cfg)
    assert run.status == 0
    err, n_near = check_router(run)
    check_layout(run)
    rng = np.random.default_rng(0)
    check_permute(run, rng.choice(cfg.nK, size=4096, replace=False))
    check_permute_scatter(run, rng.choice(cfg.nK, size=4096, replace=False))
    off = run.np("offsets")
    # rows at every expert-segment start/end and tile seams, plus random rows,
    # restricted to a few experts (the hottest, the coldest non-empty, random)
    counts = run.np("counts")
    nz = np.where(counts > 0)[0]
    pick = {int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])])}
    pick |= set(int(e) for e in rng.choice(nz, size=min(4, len(nz)), replace=False))
    rows = []
    for e in sorted(pick):
        lo, hi = off[e], off[e + 1]
        seg = np.arange(lo, hi)
        rows += list(seg[:3]) + list(seg[-3:]) + list(seg[127:130]) + list(
            rng.choice(seg, size=min(64, len(seg)), replace=False))
    check_experts(run, rows)
    check_gather_fusion(run)
    check_unweighted_gemm2_and_combine(run, rows)
    check_combine(run)
    toks = sorted(set(rng.choice(cfg.n, size=96, replace=False).tolist() + [0, cfg.n - 1]))
    check_layer(run, toks)


def test_skew_workload_is_skewed():
    run = Run(SKEW)
    counts = run.np("counts")
    cv = O.count_cv(counts)
    assert 1.35 <= cv <= 1.65, cv
    assert int((counts == 0).sum()) == 4


@pytest.mark.parametrize("E,K", [(64, 8), (256, 8), (16, 4)])
def test_router_constructed_ties(E, K):
    """Exact ties (duplicated W_gate columns) and near ties (columns one bf16
    step apart) on large-scored experts: the GPU must order them as the exact
    evaluation does, except where the oracle itself sees a gap below 1e-6."""
    import top_routing_dispatch_gb300 as M
    dev = torch.device("cuda:0")
    n, H = 1000, 256
    g = torch.Generator(device="cpu")
    g.manual_seed(E * 7 + K)
    x = torch.randn(n, H, generator=g).to(torch.bfloat16)
    wg = (torch.randn(H, E, generator=g) * 0.02)
    wg[:, [3, 5, 7, 9, 11]] *= 6.0                 # these experts score high
    wg[:, 5] = wg[:, 3]                            # exact tie 3 / 5
    wg = wg.to(torch.bfloat16)
    col = wg[:, 7].clone()
    col[::7] = torch.nextafter(col[::7].float(), torch.tensor(10.0)).to(torch.bfloat16)
    wg[:, 9] = col                                 # near tie 7 / 9 (one step apart in a few k)
    x, wg = x.to(dev), wg.to(dev)
    desc = M.make_desc(n, H, 128, E, K, "bf16", True)
    idx = torch.empty(n, K, dtype=torch.int32, device=dev)
    w = torch.empty(n, K, dtype=torch.float32, device=dev)
    logits = torch.empty(n, E, dtype=torch.float32, device=dev)
    M.moe_route_topk(desc, x, wg, None, idx, w, logits)
    torch.cuda.synchronize()
    lo = O.router_logits(f64(x), f64(wg))
    near = O.near_tie_tokens(lo, K)
    oe, ow = O.topk(lo, K, True)
    gi = idx.cpu().numpy()
    ok = ~near
    assert ok.sum() > 0
    assert np.array_equal(gi[ok], oe[ok])
    for t in np.where(near)[0]:
        assert valid_near_tie_choice(lo[t], gi[t], K)
    # exact ties resolve to the lower expert id first, as in the oracle
    both = np.array([3 in r and 5 in r for r in gi])
    assert both.any()
    for r in gi[both]:
        assert list(r).index(3) < list(r).index(5)
    ok_m, ratio, err = logit_error_within_margin(
        logits.cpu().numpy(), lo, 1e-4 * max(1.0, H / 2048.0) if E % 64 == 0 else 1e-3)
    assert ok_m, (ratio, err)
    rel = np.abs(w.cpu().numpy()[ok] - ow[ok]) / ow[ok]
    assert rel.max() <= 2.0 * err + 2e-6
