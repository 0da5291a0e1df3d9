"""The router with its weight transposed once (moe_prepare_router,
moe_layer_desc_t.w_gate_t) against the router reading W_gate as stored:
topk_idx, topk_w and logits bitwise equal -- the transposed copy only changes
where the near-tie rescoring reads each expert's column.  On constructed exact
and near ties for the warp-level MMA router (E = 64, 128), the tensor-core
router (E = 256) and the FMA router (E = 16), and at full size."""
import pytest
import torch

from workloads import DSV3, OLMOE, SKEW, synth

pytestmark = pytest.mark.gpu


def _tied(n, H, E, K, seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn(n, H, generator=g).to(torch.bfloat16)
    wg = torch.randn(H, E, generator=g) * 0.02
    wg[:, [3, 5, 7, 9, 11]] *= 6.0
    wg[:, 5] = wg[:, 3]  # exact tie
    wg = wg.to(torch.bfloat16)
    col = wg[:, 7].clone()
    col[::7] = torch.nextafter(col[::7].float(), torch.tensor(10.0)).to(torch.bfloat16)
    wg[:, 9] = col  # near tie
    return x.cuda(), wg.cuda()


def _route(M, desc, x, wg, bias, n, E, K):
    dev = x.device
    idx = torch.empty(n, K, dtype=torch.int32, device=dev)
    w = torch.empty(n, K, dtype=torch.float32, device=dev)
    logits = torch.empty(n, E, dtype=torch.float32, device=dev)
    M.moe_route_topk(desc, x, wg, bias, idx, w, logits)
    torch.cuda.synchronize()
    return idx, w, logits


def _compare(M, n, H, E, K, x, wg, bias=None, norm=True):
    desc = M.make_desc(n, H, 128, E, K, "bf16", norm)
    wgt = M.moe_prepare_router(desc, wg)
    torch.cuda.synchronize()
    assert torch.equal(wgt.view(torch.int16), wg.t().contiguous().view(torch.int16))
    a = _route(M, desc, x, wg, bias, n, E, K)
    b = _route(M, M.make_desc(n, H, 128, E, K, "bf16", norm, w_gate_t=wgt), x, wg, bias, n, E, K)
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.int32), v.view(torch.int32))


@pytest.mark.parametrize("E,K,H", [(64, 8, 256), (128, 3, 256), (256, 8, 256), (16, 4, 256),
                                   (256, 8, 7168)])
def test_router_transposed_weight_constructed_ties(E, K, H):
    import top_routing_dispatch_gb300 as M
    n = 1000
    x, wg = _tied(n, H, E, K, E * 7 + K + H)
    _compare(M, n, H, E, K, x, wg)


@pytest.mark.parametrize("cfg", [OLMOE, SKEW, DSV3], ids=lambda c: c.name)
def test_router_transposed_weight_full_size(cfg):
    import top_routing_dispatch_gb300 as M
    dev = torch.device("cuda:0")
    L = synth.make_layer(cfg, dev)
    x = synth.make_x(cfg, dev)
    _compare(M, cfg.n, cfg.H, cfg.E, cfg.K, x, L["w_gate"], L["bias"], cfg.norm_topk_prob)


def test_forward_with_transposed_router_weight():
    """The whole layer with the transposed copy in its descriptor: y bitwise
    that of the layer without it."""
    import top_routing_dispatch_gb300 as M
    from tests.gpu_helpers import Run
    run = Run(OLMOE, n=1024)
    assert run.status == 0
    wgt = M.moe_prepare_router(run.desc, run.L["w_gate"])
    layer = M.MoELayer(run.desc, run.L["w_gate"], run.L["bias"], run.L["w13"], run.L["w2"],
                       w_gate_t=wgt)
    y = layer.forward([run.x])[0]
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    assert torch.equal(y.view(torch.int16), run.y.view(torch.int16))
