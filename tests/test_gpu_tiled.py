"""Tiled expert weights (moe_prepare_weights, MOE_WEIGHTS_TILED): the layout is
the one include/moe.h states, and every expert entry point gives bitwise the
results of the row-major weights, on small shapes and at full size."""
import pytest
import torch

from tests.gpu_helpers import Run
from tests.test_gpu_parity import SMALL
from workloads import DSV3, OLMOE, SKEW

pytestmark = pytest.mark.gpu

BF16_SMALL = [c for c in SMALL if c.dtype == "bf16" and c.I % 128 == 0 and c.H % 64 == 0]


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


def _tiled_reference(w):
    """w (E, rows, cols) -> tiles ordered by expert, row block, column block,
    each 64 x 64 tile row-major: an independent restatement with torch views."""
    E, rows, cols = w.shape
    t = w.reshape(E, rows // 64, 64, cols // 64, 64).permute(0, 1, 3, 2, 4)
    return t.reshape(E, rows, cols)


def test_prepare_weights_layout():
    import top_routing_dispatch_gb300 as M
    cfg = BF16_SMALL[0]
    run = Run(cfg)
    w13t, w2t = M.moe_prepare_weights(M.desc_for(cfg), run.L["w13"], run.L["w2"])
    torch.cuda.synchronize()
    assert torch.equal(_bits(w13t), _bits(_tiled_reference(run.L["w13"])))
    assert torch.equal(_bits(w2t), _bits(_tiled_reference(run.L["w2"])))


def _check_tiled(cfg):
    import top_routing_dispatch_gb300 as M
    run = Run(cfg)
    assert run.status == 0
    desc_t = M.desc_for(cfg, tiled=True)
    w13t, w2t = M.moe_prepare_weights(M.desc_for(cfg), run.L["w13"], run.L["w2"])
    layer_t = M.MoELayer(desc_t, run.L["w_gate"], run.L["bias"], w13t, w2t)
    y_t = layer_t.forward([run.x])[0]
    torch.cuda.synchronize()
    assert int(layer_t.status.item()) == 0
    assert torch.equal(_bits(y_t), _bits(run.y))
    # the expert entry points on their own: h and the unweighted y_perm
    v = run.view
    st = torch.zeros(1, dtype=torch.int32, device=run.dev)
    h_t = torch.empty_like(v("h"))
    M.moe_expert_gemm1_swiglu(desc_t, v("x_perm"), w13t, v("offsets"), h_t, 0, st)
    assert torch.equal(_bits(h_t), _bits(layer_t.view("h")))
    h_g = torch.empty_like(v("h"))
    M.moe_expert_gemm1_swiglu_gather(desc_t, run.x, v("perm"), w13t, v("offsets"), h_g, 0, st)
    assert torch.equal(_bits(h_g), _bits(h_t))
    yp_r = torch.empty_like(v("y_perm"))
    yp_t = torch.empty_like(v("y_perm"))
    M.moe_expert_gemm2(run.desc, v("h"), run.L["w2"], v("offsets"), yp_r, 0, st)
    M.moe_expert_gemm2(desc_t, v("h"), w2t, v("offsets"), yp_t, 0, st)
    torch.cuda.synchronize()
    assert M.moe_check_status(st) == 0
    assert torch.equal(_bits(yp_t), _bits(yp_r))


@pytest.mark.parametrize("cfg", BF16_SMALL, ids=lambda c: c.name)
def test_tiled_small(cfg):
    _check_tiled(cfg)


@pytest.mark.parametrize("cfg", [OLMOE, SKEW, DSV3], ids=lambda c: c.name)
def test_tiled_full_size(cfg):
    _check_tiled(cfg)
