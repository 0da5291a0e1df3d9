"""The grouped GEMMs on CTA pairs (cta_group::2, 256-row tiles, the
default) and on single CTAs (128-row tiles, moe_set_gemm_pairs(False)) give the
same results: GEMM1 + SwiGLU (h), GEMM2 (unweighted and weighted) and the whole
layer, on the small parity shapes (one-row and ragged segments, empty experts,
segments ending in the first half of a 256-row window) and at full size.  The
oracle parity of the default path is covered by the parity tests."""
import pytest
import torch

from tests.gpu_helpers import Run
from tests.test_gpu_parity import SMALL
from workloads import DSV3, OLMOE, SKEW

pytestmark = pytest.mark.gpu

BF16_SMALL = [c for c in SMALL if c.dtype == "bf16"]


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


def _gemms(M, run, st, sm_reserve):
    v = run.view
    h = torch.empty_like(v("h"))
    yp = torch.empty_like(v("y_perm"))
    ys = torch.empty_like(v("y_perm"))
    M.moe_expert_gemm1_swiglu(run.desc, v("x_perm"), run.L["w13"], v("offsets"), h, sm_reserve,
                              st)
    M.moe_expert_gemm2(run.desc, v("h"), run.L["w2"], v("offsets"), yp, sm_reserve, st)
    M.moe_expert_gemm2_weighted(run.desc, v("h"), run.L["w2"], v("offsets"), v("perm"),
                                v("topk_w"), ys, sm_reserve, st)
    return h, yp, ys


def _check(cfg, sm_reserve=0):
    import top_routing_dispatch_gb300 as M
    M.moe_set_gemm_pairs(True)
    run = Run(cfg)  # forward on CTA pairs
    assert run.status == 0
    st = torch.zeros(1, dtype=torch.int32, device=run.dev)
    pair = _gemms(M, run, st, sm_reserve)
    try:
        M.moe_set_gemm_pairs(False)
        single = _gemms(M, run, st, sm_reserve)
        y1 = run.layer.forward([run.x])[0].clone()
    finally:
        M.moe_set_gemm_pairs(True)
    torch.cuda.synchronize()
    assert M.moe_check_status(st) == 0
    assert int(run.layer.status.item()) == 0
    for name, a, b in zip(("h", "y_perm", "y_slot"), pair, single):
        assert torch.equal(_bits(a), _bits(b)), name
    # the forward's own intermediates came from the pair kernels
    assert torch.equal(_bits(pair[0]), _bits(run.view("h")))
    assert torch.equal(_bits(y1), _bits(run.y))


@pytest.mark.parametrize("cfg", BF16_SMALL, ids=lambda c: c.name)
def test_pairs_small(cfg):
    _check(cfg)


def test_pairs_sm_reserve():
    # fewer resident pairs than SMs / 2: the tile loop strides by the pair count
    _check(BF16_SMALL[0], sm_reserve=100)


@pytest.mark.parametrize("cfg", [OLMOE, SKEW, DSV3], ids=lambda c: c.name)
def test_pairs_full_size(cfg):
    _check(cfg)


@pytest.mark.parametrize("name", ["bwd_bf16", "bwd_skew_e64", "bwd_e128", "olmoe"])
def test_pairs_backward(name):
    """moe_backward's dgrad (K-major weight operand) and SwiGLU-backward GEMMs
    on CTA pairs against single CTAs: every gradient bitwise equal."""
    import top_routing_dispatch_gb300 as M
    from tests.test_gpu_backward import CASES, _run
    cfg = OLMOE if name == "olmoe" else next(c for c in CASES if c.name == name)
    M.moe_set_gemm_pairs(True)
    a = _run(cfg)
    try:
        M.moe_set_gemm_pairs(False)
        b = _run(cfg)
    finally:
        M.moe_set_gemm_pairs(True)
    assert a["status"] == 0 and b["status"] == 0
    for k in ("dx", "dwg", "dbias", "dw13", "dw2"):
        assert torch.equal(a[k].view(torch.uint8), b[k].view(torch.uint8)), k
