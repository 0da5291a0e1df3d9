"""Two-stream micro-batch schedule and edge cases, through the C ABI."""
import numpy as np
import pytest
import torch

import top_routing_dispatch_gb300 as M
from oracle import moe_oracle as O
from tests.gpu_helpers import TOL, rel_fro, f64
from workloads import DOMINO, synth
from workloads.configs import MoEConfig

pytestmark = pytest.mark.gpu


def _layer(cfg, num_mb):
    dev = torch.device("cuda:0")
    L = synth.make_layer(cfg, dev)
    return L, M.MoELayer(M.desc_for(cfg), L["w_gate"], L["bias"], L["w13"], L["w2"],
                         num_mb=num_mb)


def test_two_stream_equals_sequential_bitwise():
    cfg = DOMINO
    dev = torch.device("cuda:0")
    L, two = _layer(cfg, 2)
    xs = synth.make_micro_batches(cfg, dev)
    sc = torch.cuda.Stream()
    sd = torch.cuda.Stream()
    torch.cuda.synchronize()
    ys2 = two.forward(xs, sm_reserve=16, compute=sc, dispatch=sd)
    torch.cuda.synchronize()
    two.check()
    one = M.MoELayer(M.desc_for(cfg), L["w_gate"], L["bias"], L["w13"], L["w2"])
    seq = [one(x).clone() for x in xs]
    torch.cuda.synchronize()
    for a, b in zip(ys2, seq):
        assert torch.equal(a, b)
    # each micro-batch against the oracle on sampled tokens
    rng = np.random.default_rng(1)
    for x, y in zip(xs, ys2):
        toks = np.sort(rng.choice(cfg.n, size=64, replace=False))
        ti = torch.as_tensor(toks, device=dev)
        r = O.moe_forward(f64(x[ti]), f64(L["w_gate"]), None, lambda e: f64(L["w13"][e]),
                          lambda e: f64(L["w2"][e]), cfg.K, cfg.norm_topk_prob)
        assert rel_fro(f64(y[ti]), r["y"]) <= TOL["bf16"]


def test_four_micro_batches_two_streams_bitwise():
    """Four micro-batches through the two-stream schedule (every cross-batch
    dependency of the pipeline used more than once) equal four single-stream
    calls bit for bit."""
    cfg = MoEConfig("mb4_bf16", n=512, H=2048, I=1024, E=64, K=8, dtype="bf16",
                    norm_topk_prob=False, seed=36)
    dev = torch.device("cuda:0")
    L, four = _layer(cfg, 4)
    xs = [synth.make_x(cfg, dev, seed=60 + i) for i in range(4)]
    sc, sd = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    ys = four.forward(xs, compute=sc, dispatch=sd)
    torch.cuda.synchronize()
    four.check()
    one = M.MoELayer(M.desc_for(cfg), L["w_gate"], L["bias"], L["w13"], L["w2"])
    for x, y in zip(xs, ys):
        assert torch.equal(one(x), y)


@pytest.mark.parametrize("reserve", [8, 40, 140])
def test_sm_reserve_does_not_change_results(reserve):
    cfg = MoEConfig("reserve_bf16", n=700, H=256, I=256, E=8, K=2, dtype="bf16",
                    norm_topk_prob=False, seed=31)
    dev = torch.device("cuda:0")
    _, layer = _layer(cfg, 1)
    x = synth.make_x(cfg, dev)
    y0 = layer.forward([x])[0].clone()
    y1 = layer.forward([x], sm_reserve=reserve)[0].clone()
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)


def test_repeated_calls_reuse_buffers():
    cfg = MoEConfig("reuse_bf16", n=257, H=128, I=128, E=6, K=2, dtype="bf16",
                    norm_topk_prob=True, seed=32)
    dev = torch.device("cuda:0")
    _, layer = _layer(cfg, 1)
    x1 = synth.make_x(cfg, dev, seed=1)
    x2 = synth.make_x(cfg, dev, seed=2)
    a = layer(x1).clone()
    b = layer(x2).clone()
    c = layer(x1).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, c)
    assert not torch.equal(a, b)


def test_zero_tokens():
    cfg = MoEConfig("empty_bf16", n=0, H=128, I=128, E=4, K=2, dtype="bf16",
                    norm_topk_prob=False, seed=33)
    dev = torch.device("cuda:0")
    _, layer = _layer(cfg, 1)
    x = torch.empty((0, 128), dtype=torch.bfloat16, device=dev)
    y = layer(x)
    torch.cuda.synchronize()
    layer.check()
    assert y.shape == (0, 128)
    assert layer.view("offsets").cpu().tolist() == [0] * 5


def _layout(desc, idx):
    dev = idx.device
    nK = idx.numel()
    E = desc.E
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(nK, dtype=torch.int32, device=dev)
    inv = torch.empty(nK, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(max(M.moe_layout_workspace_size(desc), 1), dtype=torch.uint8, device=dev)
    M.moe_dispatch_layout(desc, idx, counts, offsets, perm, inv, status, ws)
    st = M.moe_check_status(status)
    return st, counts.cpu().numpy(), offsets.cpu().numpy(), perm.cpu().numpy(), inv.cpu().numpy()


def test_layout_printed_example():
    """The moe_align_block_size example (ids shifted to 0-based) on the GPU."""
    idx = torch.tensor([[2, 3, 4], [1, 2, 4], [1, 3, 4], [1, 2, 3]], dtype=torch.int32,
                       device="cuda:0") - 1
    desc = M.make_desc(4, 64, 128, 4, 3, "bf16", False)
    st, counts, offsets, perm, inv = _layout(desc, idx)
    assert st == 0
    assert counts.tolist() == [3, 3, 3, 3]
    assert offsets.tolist() == [0, 3, 6, 9, 12]
    assert perm.tolist() == [3, 6, 9, 0, 4, 10, 1, 7, 11, 2, 5, 8]


# n*K <= 65536 runs the single-CTA layout, above it the three-kernel layout
@pytest.mark.parametrize("n,E,K,hot", [(5000, 64, 8, False), (3001, 256, 8, True),
                                       (4096, 1, 1, False), (1, 7, 3, False),
                                       (8192, 64, 8, False), (8193, 64, 8, False),
                                       (20000, 256, 8, True)])
def test_layout_edge_shapes(n, E, K, hot):
    g = torch.Generator(device="cpu")
    g.manual_seed(n * 31 + E)
    idx = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(n)]).to(torch.int32)
    if hot:
        idx[: n // 2, 0] = 3            # one hot expert; others may be empty
        idx[: n // 2, 1:] = torch.arange(4, 4 + K - 1, dtype=torch.int32)
    desc = M.make_desc(n, 64, 128, E, K, "bf16", False)
    st, counts, offsets, perm, inv = _layout(desc, idx.cuda())
    assert st == 0
    oc, oo, op, oi = O.dispatch_layout(idx.numpy(), E)
    assert np.array_equal(counts, oc) and np.array_equal(offsets, oo)
    assert np.array_equal(perm, op) and np.array_equal(inv, oi)


def test_layout_bad_ids_flagged_and_perm_stays_a_permutation():
    idx = torch.tensor([[0, 1], [5, 2], [-1, 3], [2, 9]], dtype=torch.int32, device="cuda:0")
    desc = M.make_desc(4, 64, 128, 4, 2, "bf16", False)
    st, counts, offsets, perm, inv = _layout(desc, idx)
    assert st == 4  # MOE_ERR_BAD_ROUTING
    assert sorted(perm.tolist()) == list(range(8))
    assert offsets[-1] == 5                       # five valid pairs
    assert counts.tolist() == [1, 1, 2, 1]
    assert np.array_equal(inv[perm], np.arange(8))


@pytest.mark.parametrize("n", [3000, 9000])
def test_layout_bad_ids_both_paths(n):
    """Invalid ids on the single-CTA (n*K <= 65536) and the multi-block path:
    flagged, valid pairs laid out as the oracle lays out the valid subset,
    invalid pairs after them in ascending flat index."""
    E, K = 16, 8
    g = torch.Generator(device="cpu")
    g.manual_seed(n)
    idx = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(n)]).to(torch.int32)
    bad = torch.rand(idx.shape, generator=g) < 0.01
    idx[bad] = torch.where(torch.rand(idx.shape, generator=g)[bad] < 0.5, -1, E + 3).to(torch.int32)
    desc = M.make_desc(n, 64, 128, E, K, "bf16", False)
    st, counts, offsets, perm, inv = _layout(desc, idx.cuda())
    assert st == 4  # MOE_ERR_BAD_ROUTING
    flat = idx.numpy().reshape(-1)
    ok = (flat >= 0) & (flat < E)
    nv = int(ok.sum())
    assert offsets[-1] == nv
    assert counts.tolist() == np.bincount(flat[ok], minlength=E).tolist()
    valid_f = np.where(ok)[0]
    order = valid_f[np.argsort(flat[ok], kind="stable")]
    assert np.array_equal(perm[:nv], order)
    assert np.array_equal(perm[nv:], np.where(~ok)[0])
    assert np.array_equal(inv[perm], np.arange(n * K))
