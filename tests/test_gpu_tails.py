"""Fused tails of the CTA-pair grouped GEMMs: an expert whose rows end 1..32
rows past a 256-row window boundary (after at least one full window) computes
those rows inside its last full window's tiles, transposed (the weight columns
as the 256-row operand, the tail rows as a 32-column one).  Segment lengths on
both sides of every boundary of that rule (an empty expert, one row, 256 + 1,
256 + 32, 256 + 33, 512 + 1, ..., the last segment's tail ending at the last
row, so that the odd CTA's tail rows lie past the tensor) give bitwise the
results without fused tails and those of single CTAs, for GEMM1 + SwiGLU and
both GEMM2 forms, every output row is written, and h, y_perm and y_slot match the oracle's expert steps
(Algorithm 2 steps 8-9 of "MoE 分布式推理基础（基于 vLLM）" §1.2).  The
pipeline-wait timeout leaves tiles with tails cleanly too."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from tests.gpu_helpers import TOL, f64, rel_fro

pytestmark = pytest.mark.gpu

LENS = [257, 1, 288, 289, 0, 256, 270, 31, 512, 513, 544, 545, 800, 801, 300, 192, 768,
        260]


def _inputs(H, I, lens, seed):
    g = torch.Generator().manual_seed(seed)
    E, nK = len(lens), int(sum(lens))
    x = torch.randn(nK, H, generator=g).to(torch.bfloat16)
    w13 = (torch.randn(E, H, 2 * I, generator=g) * H ** -0.5).to(torch.bfloat16)
    w2 = (torch.randn(E, I, H, generator=g) * I ** -0.5).to(torch.bfloat16)
    off = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    perm = torch.randperm(nK, generator=g).to(torch.int32)
    tw = torch.rand(nK, generator=g)
    dev = torch.device("cuda:0")
    return [t.to(dev) for t in (x, w13, w2, off, perm, tw)]


def _gemms(M, desc, x, w13, w2, off, perm, tw, h_in, st):
    nK, H = x.shape
    I = w2.shape[1]
    nan = float("nan")  # rows a kernel missed keep it, and differ from the other form's
    h = torch.full((nK, I), nan, dtype=torch.bfloat16, device=x.device)
    yp = torch.full((nK, H), nan, dtype=torch.bfloat16, device=x.device)
    ys = torch.full((nK, H), nan, dtype=torch.bfloat16, device=x.device)
    M.moe_expert_gemm1_swiglu(desc, x, w13, off, h, 0, st)
    src = h if h_in is None else h_in
    M.moe_expert_gemm2(desc, src, w2, off, yp, 0, st)
    M.moe_expert_gemm2_weighted(desc, src, w2, off, perm, tw, ys, 0, st)
    return h, yp, ys


@pytest.mark.parametrize("H,I", [(320, 256), (2048, 1024)], ids=["h320_i256", "h2048_i1024"])
def test_fused_tails(H, I):
    import top_routing_dispatch_gb300 as M
    x, w13, w2, off, perm, tw = _inputs(H, I, LENS, seed=11)
    nK = x.shape[0]
    desc = M.make_desc(nK, H, I, len(LENS), 1, "bf16", False)
    st = torch.zeros(1, dtype=torch.int32, device=x.device)
    M.moe_set_gemm_pairs(True)
    try:
        M.moe_set_gemm_tails(True)
        pair = _gemms(M, desc, x, w13, w2, off, perm, tw, None, st)
        M.moe_set_gemm_tails(False)
        pair_nt = _gemms(M, desc, x, w13, w2, off, perm, tw, pair[0], st)
        M.moe_set_gemm_pairs(False)
        single = _gemms(M, desc, x, w13, w2, off, perm, tw, pair[0], st)
    finally:
        M.moe_set_gemm_pairs(True)
        M.moe_set_gemm_tails(None)
    torch.cuda.synchronize()
    assert M.moe_check_status(st) == 0
    for name, a, b, c in zip(("h", "y_perm", "y_slot"), pair, pair_nt, single):
        assert not torch.isnan(a.float()).any(), name
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name
        assert torch.equal(a.view(torch.int16), c.view(torch.int16)), name
    # the oracle's expert steps on the same inputs (y from the GPU's own h)
    h, yp, ys = (f64(t) for t in pair)
    xs, hs = f64(x), f64(pair[0])
    o = off.cpu().numpy()
    p = perm.cpu().numpy()
    twn = tw.double().cpu().numpy()
    for e in range(len(LENS)):
        lo, hi = int(o[e]), int(o[e + 1])
        if hi == lo:
            continue
        h_ref = O.expert_up(xs[lo:hi], f64(w13[e]))
        y_ref = O.expert_down(hs[lo:hi], f64(w2[e]))
        assert rel_fro(h[lo:hi], h_ref) < TOL["bf16"], e
        assert rel_fro(yp[lo:hi], y_ref) < TOL["bf16"], e
        assert rel_fro(ys[p[lo:hi]], twn[p[lo:hi], None] * y_ref) < TOL["bf16"], e


def test_fused_tails_timeout_recovers():
    """Waits limited to 200 cycles: GEMM1 and the weighted GEMM2 give up with
    MOE_ERR_TIMEOUT (the gate and up warps of a tail agree to stop together,
    the leader settles the half-loaded stages with their tail bytes); the next
    calls, with the default limit, give the same bits as before."""
    import top_routing_dispatch_gb300 as M
    MOE_ERR_TIMEOUT = 6
    H, I = 2048, 1024
    x, w13, w2, off, perm, tw = _inputs(H, I, LENS, seed=12)
    nK = x.shape[0]
    desc = M.make_desc(nK, H, I, len(LENS), 1, "bf16", False)
    st = torch.zeros(1, dtype=torch.int32, device=x.device)
    M.moe_set_gemm_pairs(True)
    M.moe_set_gemm_tails(True)
    try:
        ref = _gemms(M, desc, x, w13, w2, off, perm, tw, None, st)
        torch.cuda.synchronize()
        assert M.moe_check_status(st) == 0
        try:
            M.moe_set_pipeline_wait_limit(200)
            st.zero_()
            _gemms(M, desc, x, w13, w2, off, perm, tw, None, st)
            got = M.moe_check_status(st)
        finally:
            M.moe_set_pipeline_wait_limit(0)
        assert got == MOE_ERR_TIMEOUT
        st.zero_()
        again = _gemms(M, desc, x, w13, w2, off, perm, tw, None, st)
        torch.cuda.synchronize()
    finally:
        M.moe_set_gemm_tails(None)
    assert M.moe_check_status(st) == 0
    for name, a, b in zip(("h", "y_perm", "y_slot"), again, ref):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name


@pytest.mark.parametrize("name", ["olmoe", "olmoe_tiled"])
def test_fused_tails_forced_full_size(name):
    """The OLMoE-shaped layer (512 rows per expert on average: tails are off
    by default there) with fused tails forced on, row-major and tiled
    weights: the layer output and h bitwise equal to the default path."""
    import top_routing_dispatch_gb300 as M
    from tests.gpu_helpers import Run
    from workloads import OLMOE
    run = Run(OLMOE)
    assert run.status == 0
    tiled = name.endswith("tiled")
    if tiled:
        desc = M.desc_for(OLMOE, tiled=True)
        w13, w2 = M.moe_prepare_weights(M.desc_for(OLMOE), run.L["w13"], run.L["w2"])
    else:
        desc, w13, w2 = run.desc, run.L["w13"], run.L["w2"]
    layer = M.MoELayer(desc, run.L["w_gate"], run.L["bias"], w13, w2)
    try:
        M.moe_set_gemm_tails(True)
        y = layer.forward([run.x])[0]
        torch.cuda.synchronize()
    finally:
        M.moe_set_gemm_tails(None)
    assert int(layer.status.item()) == 0
    assert torch.equal(y.view(torch.int16), run.y.view(torch.int16))
    assert torch.equal(layer.view("h").view(torch.int16), run.view("h").view(torch.int16))
