"""GPU backward (moe_backward) against the fp64 backward oracle
(oracle/moe_backward.py) on the same seeded inputs, through the C ABI.
The forward intermediates come from the library's own entry points (router,
layout, permute, GEMM1 + SwiGLU, unweighted GEMM2); near-tie tokens use the
GPU's expert choice in the oracle, as the forward parity tests do."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from oracle import moe_backward as OB
from tests.gpu_helpers import NEAR_TIE_GAP, rel_fro, f64
from workloads import synth
from workloads.configs import MoEConfig

pytestmark = pytest.mark.gpu

CASES = [
    MoEConfig("bwd_bf16", n=384, H=256, I=128, E=8, K=2, dtype="bf16", norm_topk_prob=True,
              seed=41),
    MoEConfig("bwd_skew_e64", n=600, H=512, I=256, E=64, K=6, dtype="bf16",
              norm_topk_prob=False, seed=42, skew=True),
    MoEConfig("bwd_one_token", n=1, H=256, I=128, E=8, K=2, dtype="bf16", norm_topk_prob=True,
              seed=43),
    # K = 12 (the 16-slot kernels), E = 20 (not a multiple of 8; the FMA router)
    MoEConfig("bwd_k12", n=150, H=256, I=128, E=32, K=12, dtype="bf16", norm_topk_prob=True,
              seed=45),
    MoEConfig("bwd_e20", n=300, H=512, I=384, E=20, K=3, dtype="bf16", norm_topk_prob=False,
              seed=46),
    # E = 128: two 64-expert tiles in dW_gate and the router's tensor-core path
    MoEConfig("bwd_e128", n=400, H=256, I=128, E=128, K=4, dtype="bf16", norm_topk_prob=True,
              seed=49),
]
TOL = 2e-2


def _run(cfg, force=None):
    """Forward intermediates from the library's entry points, then
    moe_backward.  `force` (n, K) replaces the router's expert choice (the
    weights are then the softmax of the router's logits at those experts)."""
    import top_routing_dispatch_gb300 as M
    dev = torch.device("cuda:0")
    L = synth.make_layer(cfg, dev)
    x = synth.make_x(cfg, dev)
    g = torch.Generator(device=dev)
    g.manual_seed(synth.sub_seed(cfg.seed, "dy"))
    dy = torch.randn((cfg.n, cfg.H), generator=g, device=dev).to(torch.bfloat16)
    desc = M.desc_for(cfg)
    n, H, I, E, K, nK = cfg.n, cfg.H, cfg.I, cfg.E, cfg.K, cfg.nK
    i32, f32, bf = torch.int32, torch.float32, torch.bfloat16
    logits = torch.empty((n, E), dtype=f32, device=dev)
    idx = torch.empty((n, K), dtype=i32, device=dev)
    w = torch.empty((n, K), dtype=f32, device=dev)
    counts = torch.empty(E, dtype=i32, device=dev)
    offsets = torch.empty(E + 1, dtype=i32, device=dev)
    perm = torch.empty(nK, dtype=i32, device=dev)
    inv = torch.empty(nK, dtype=i32, device=dev)
    st = torch.zeros(1, dtype=i32, device=dev)
    lws = torch.empty(max(M.moe_layout_workspace_size(desc), 1), dtype=torch.uint8, device=dev)
    xp = torch.empty((nK, H), dtype=bf, device=dev)
    h = torch.empty((nK, I), dtype=bf, device=dev)
    yp = torch.empty((nK, H), dtype=bf, device=dev)
    M.moe_route_topk(desc, x, L["w_gate"], L["bias"], idx, w, logits)
    if force is not None:
        idx.copy_(torch.as_tensor(force, dtype=i32, device=dev))
        p = torch.softmax(logits.double(), dim=1).gather(1, idx.long())
        if cfg.norm_topk_prob:
            p = p / p.sum(dim=1, keepdim=True)
        w.copy_(p.float())
    M.moe_dispatch_layout(desc, idx, counts, offsets, perm, inv, st, lws)
    M.moe_permute(desc, x, perm, xp, st)
    M.moe_expert_gemm1_swiglu(desc, xp, L["w13"], offsets, h, status_word=st)
    M.moe_expert_gemm2(desc, h, L["w2"], offsets, yp, status_word=st)
    dx = torch.empty_like(x)
    dwg = torch.empty((H, E), dtype=f32, device=dev)
    dbias = torch.empty(E, dtype=f32, device=dev)
    dw13 = torch.empty((E, H, 2 * I), dtype=f32, device=dev)
    dw2 = torch.empty((E, I, H), dtype=f32, device=dev)
    ws = torch.empty(M.moe_backward_workspace_size(desc), dtype=torch.uint8, device=dev)
    M.moe_backward(desc, x, L["w_gate"], L["w13"], L["w2"], dy, logits, idx, w, offsets, inv, xp,
                   h, yp, dx, dwg, dbias, dw13, dw2, ws, st)
    torch.cuda.synchronize()
    return dict(L=L, x=x, dy=dy, idx=idx, status=int(st.item()), dx=dx, dwg=dwg, dbias=dbias,
                dw13=dw13, dw2=dw2, counts=counts.cpu().numpy())


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_backward_matches_oracle(cfg):
    r = _run(cfg)
    assert r["status"] == 0
    L = r["L"]
    x64 = f64(r["x"])
    wg64 = f64(L["w_gate"])
    b64 = f64(L["bias"])
    lo = O.router_logits(x64, wg64, b64)
    near = O.near_tie_tokens(lo, cfg.K, NEAR_TIE_GAP)
    gidx = r["idx"].cpu().numpy()
    forced = (np.where(near)[0], gidx[near])
    w13 = lambda e: L["w13"][e].to(torch.float64).cpu().numpy()
    w2 = lambda e: L["w2"][e].to(torch.float64).cpu().numpy()
    o = OB.moe_backward(x64, wg64, b64, w13, w2, cfg.K, cfg.norm_topk_prob, f64(r["dy"]),
                        forced=forced)
    errs = dict(dx=rel_fro(f64(r["dx"]), o["dx"]),
                dw_gate=rel_fro(f64(r["dwg"]), o["dw_gate"]),
                dw13=rel_fro(f64(r["dw13"]), o["dw13"]),
                dw2=rel_fro(f64(r["dw2"]), o["dw2"]))
    if cfg.skew:
        errs["dbias"] = rel_fro(f64(r["dbias"]), o["dbias"])
    print(cfg.name, {k: f"{v:.2e}" for k, v in errs.items()})
    for k, v in errs.items():
        assert v <= TOL, (k, v)


def test_backward_is_deterministic():
    cfg = CASES[0]
    a, b = _run(cfg), _run(cfg)
    for k in ("dx", "dwg", "dbias", "dw13", "dw2"):
        assert torch.equal(a[k].view(torch.uint8), b[k].view(torch.uint8)), k


def test_backward_full_size_sampled():
    """The OLMoE-shaped layer (n=4096, H=2048, I=1024, E=64, K=8): dW_gate and
    the routing-weight gradients for every token; dx for sampled tokens
    (the expert backward is row-local); dW13 and dW2 for three experts (the
    hottest, the coldest, one at random) over all of their rows."""
    from workloads import OLMOE
    cfg = OLMOE
    r = _run(cfg)
    assert r["status"] == 0
    L = r["L"]
    K = cfg.K
    x64, wg64, dy64 = f64(r["x"]), f64(L["w_gate"]), f64(r["dy"])
    lo = O.router_logits(x64, wg64, None)
    near = O.near_tie_tokens(lo, K, NEAR_TIE_GAP)
    gidx = r["idx"].cpu().numpy()
    forced = (np.where(near)[0], gidx[near])
    w13 = lambda e: L["w13"][e].to(torch.float64).cpu().numpy()
    w2 = lambda e: L["w2"][e].to(torch.float64).cpu().numpy()
    fw = O.moe_forward(x64, wg64, None, w13, w2, K, cfg.norm_topk_prob, forced=forced)
    dY, dw = OB.combine_backward(dy64, fw["y_perm"], fw["w_top"], fw["inv_perm"])
    dl, dx_router, dwg = OB.router_backward(x64, wg64, fw["logits"], fw["e_top"], fw["w_top"],
                                            dw, cfg.norm_topk_prob)
    assert rel_fro(f64(r["dwg"]), dwg) <= TOL
    # dx for sampled tokens, from their K rows
    rng = np.random.default_rng(0)
    toks = np.unique(np.concatenate([rng.choice(cfg.n, 48, replace=False), [0, cfg.n - 1]]))
    inv = fw["inv_perm"].reshape(cfg.n, K)
    off = fw["offsets"]
    x_perm = O.permute(x64, fw["perm"], K)
    dx_ref = dx_router[toks].copy()
    for i, t in enumerate(toks):
        for k in range(K):
            row = inv[t, k]
            e = int(np.searchsorted(off, row, side="right") - 1)
            b = OB.expert_backward(x_perm[row:row + 1], w13(e), w2(e), dY[row:row + 1])
            dx_ref[i] += b["dX"][0]
    assert rel_fro(f64(r["dx"][torch.as_tensor(toks, device=r["dx"].device)]), dx_ref) <= TOL
    # weight gradients of three experts
    counts = np.diff(off)
    nz = np.where(counts > 0)[0]
    experts = {int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])]),
               int(rng.choice(nz))}
    for e in sorted(experts):
        lo_, hi_ = int(off[e]), int(off[e + 1])
        b = OB.expert_backward(x_perm[lo_:hi_], w13(e), w2(e), dY[lo_:hi_])
        assert rel_fro(f64(r["dw13"][e]), b["dW13"]) <= TOL, e
        assert rel_fro(f64(r["dw2"][e]), b["dW2"]) <= TOL, e


def test_backward_segment_lengths_at_block_edges():
    """Expert segments of 0, 1, 16, 17, 48, 64, 65 and 129 rows (forced
    routing, K = 1): whole and partial 16-row k steps, whole and partial
    64-row blocks, an empty expert.  The weight gradients are sums over each
    segment's rows only; rows of the neighbouring expert must not leak in."""
    counts = np.array([0, 16, 48, 64, 65, 17, 1, 129])
    cfg = MoEConfig("bwd_edges", n=int(counts.sum()), H=256, I=128, E=8, K=1, dtype="bf16",
                    norm_topk_prob=False, seed=44)
    rng = np.random.default_rng(44)
    ids = rng.permutation(np.repeat(np.arange(cfg.E), counts))[:, None]
    r = _run(cfg, force=ids)
    assert r["status"] == 0
    assert np.array_equal(r["counts"], counts)
    L = r["L"]
    x64, wg64, b64 = f64(r["x"]), f64(L["w_gate"]), f64(L["bias"])
    w13 = lambda e: L["w13"][e].to(torch.float64).cpu().numpy()
    w2 = lambda e: L["w2"][e].to(torch.float64).cpu().numpy()
    o = OB.moe_backward(x64, wg64, b64, w13, w2, 1, False, f64(r["dy"]),
                        forced=(np.arange(cfg.n), ids))
    assert np.all(f64(r["dw13"][0]) == 0) and np.all(f64(r["dw2"][0]) == 0)
    for e in range(1, cfg.E):
        assert rel_fro(f64(r["dw13"][e]), o["dw13"][e]) <= TOL, e
        assert rel_fro(f64(r["dw2"][e]), o["dw2"][e]) <= TOL, e
    assert rel_fro(f64(r["dx"]), o["dx"]) <= TOL
    assert rel_fro(f64(r["dwg"]), o["dw_gate"]) <= TOL


def test_backward_zero_tokens():
    """No tokens: every weight gradient is zero; token arrays may be empty."""
    import top_routing_dispatch_gb300 as M
    cfg = MoEConfig("bwd_empty", n=0, H=256, I=128, E=8, K=2, dtype="bf16", norm_topk_prob=True,
                    seed=47)
    dev = torch.device("cuda:0")
    L = synth.make_layer(cfg, dev)
    desc = M.desc_for(cfg)
    e = lambda shape, dt: torch.full(shape, 7.0, dtype=dt, device=dev)
    none = torch.empty(0, dtype=torch.bfloat16, device=dev)
    dwg, dbias = e((cfg.H, cfg.E), torch.float32), e((cfg.E,), torch.float32)
    dw13 = e((cfg.E, cfg.H, 2 * cfg.I), torch.float32)
    dw2 = e((cfg.E, cfg.I, cfg.H), torch.float32)
    M.moe_backward(desc, none, L["w_gate"], L["w13"], L["w2"], none, none, none, none, none,
                   none, none, none, none, none, dwg, dbias, dw13, dw2, none)
    torch.cuda.synchronize()
    for t in (dwg, dbias, dw13, dw2):
        assert int(torch.count_nonzero(t)) == 0


def test_backward_single_renormalised_slot_router_gradient_is_zero():
    """K = 1 with renormalisation: the weight is 1 for every logit vector, so
    dW_gate and dbias are exactly zero (dp = (dw - dw * 1) / p = 0 in float32
    too); the expert gradients still match the oracle."""
    cfg = MoEConfig("bwd_k1_norm", n=256, H=256, I=128, E=8, K=1, dtype="bf16",
                    norm_topk_prob=True, seed=48)
    r = _run(cfg)
    assert r["status"] == 0
    assert int(torch.count_nonzero(r["dwg"])) == 0
    assert int(torch.count_nonzero(r["dbias"])) == 0
    L = r["L"]
    x64, wg64, b64 = f64(r["x"]), f64(L["w_gate"]), f64(L["bias"])
    near = O.near_tie_tokens(O.router_logits(x64, wg64, b64), cfg.K, NEAR_TIE_GAP)
    forced = (np.where(near)[0], r["idx"].cpu().numpy()[near])
    o = OB.moe_backward(x64, wg64, b64, lambda e: L["w13"][e].to(torch.float64).cpu().numpy(),
                        lambda e: L["w2"][e].to(torch.float64).cpu().numpy(), 1, True,
                        f64(r["dy"]), forced=forced)
    assert rel_fro(f64(r["dw13"]), o["dw13"]) <= TOL
    assert rel_fro(f64(r["dx"]), o["dx"]) <= TOL
