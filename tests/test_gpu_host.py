"""moe_forward_host: the layer on pinned host buffers, copies of consecutive
calls overlapped with their neighbours' layers.  Every call's y must equal
the device-buffer forward on the same input, bit for bit."""
import pytest
import torch

from workloads import synth, TINY
from workloads.configs import MoEConfig

pytestmark = pytest.mark.gpu

CASES = [
    MoEConfig("host_bf16", n=700, H=256, I=256, E=16, K=4, dtype="bf16", norm_topk_prob=True,
              seed=31),
    MoEConfig("host_e64_bf16", n=1500, H=512, I=256, E=64, K=8, dtype="bf16",
              norm_topk_prob=False, seed=32),
    TINY,
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_forward_host_matches_device_forward(cfg):
    import top_routing_dispatch_gb300 as M
    dev = torch.device("cuda:0")
    L = synth.make_layer(cfg, dev)
    desc = M.desc_for(cfg)
    layer = M.MoELayer(desc, L["w_gate"], L["bias"], L["w13"], L["w2"])
    xs = [synth.make_x(cfg, dev, seed=100 + i) for i in range(5)]
    ref = [layer.forward([x])[0].clone() for x in xs]
    torch.cuda.synchronize()
    layer.check()
    pipe = M.HostPipeline(layer)
    xh = [x.cpu().pin_memory() for x in xs]
    yh = [torch.full_like(h, float("nan")).pin_memory() for h in xh]
    for i in range(len(xs)):            # slots 0, 1, 0, 1, 0: each slot reused
        pipe(xh[i], yh[i])
    pipe.synchronize()
    torch.cuda.synchronize()
    layer.check()
    for i in range(len(xs)):
        assert torch.equal(yh[i].view(torch.uint8), ref[i].cpu().view(torch.uint8)), i
