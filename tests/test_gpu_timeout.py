"""The device timeout path of the tensor-core GEMMs, exercised without a GPU
fault: the pipeline waits are given a limit of a few hundred cycles (far below
the time a tile's first operands take to arrive), so they give up.  The call
must report MOE_ERR_TIMEOUT through the status word, every CTA must leave
cleanly (the drain waits keep their full limit), and the next call on the same
device, with the default limit back, must compute the same result as before."""
import pytest
import torch

from tests.gpu_helpers import Run
from workloads import OLMOE

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = 6


def _gemm1(M, run, h, st):
    v = run.view
    M.moe_expert_gemm1_swiglu(run.desc, v("x_perm"), run.L["w13"], v("offsets"), h, 0, st)


@pytest.mark.parametrize("pairs", [True, False], ids=["cta_pairs", "single_cta"])
def test_pipeline_wait_timeout_reports_and_recovers(pairs):
    """CTA pairs: both CTAs give up on their own; the leader settles the
    stages whose two halves were not both loaded before the pair leaves."""
    import top_routing_dispatch_gb300 as M
    run = Run(OLMOE, n=512)
    assert run.status == 0
    st = torch.zeros(1, dtype=torch.int32, device=run.dev)
    ref = torch.empty_like(run.view("h"))
    _gemm1(M, run, ref, st)
    assert M.moe_check_status(st) == 0
    try:
        M.moe_set_gemm_pairs(pairs)
        M.moe_set_pipeline_wait_limit(200)
        h = torch.zeros_like(ref)
        st.zero_()
        _gemm1(M, run, h, st)
        got = M.moe_check_status(st)
    finally:
        M.moe_set_pipeline_wait_limit(0)
        M.moe_set_gemm_pairs(True)
    assert got == MOE_ERR_TIMEOUT
    # the context is usable and the default limit is back: same bits as before
    st.zero_()
    h2 = torch.empty_like(ref)
    _gemm1(M, run, h2, st)
    assert M.moe_check_status(st) == 0
    assert torch.equal(h2.view(torch.int16), ref.view(torch.int16))
    # and the whole layer still matches its first run
    y = run.layer.forward([run.x])[0]
    torch.cuda.synchronize()
    assert int(run.layer.status.item()) == 0
    assert torch.equal(y.view(torch.int16), run.y.view(torch.int16))


@pytest.mark.parametrize("pairs", [True, False], ids=["cta_pairs", "single_cta"])
def test_backward_timeout_reports_and_recovers(pairs):
    """The backward's GEMMs (dgrad, SwiGLU backward, weight gradients) give up
    the same way; a normal call afterwards gives the same bits as before."""
    import top_routing_dispatch_gb300 as M
    from tests.test_gpu_backward import CASES, _run
    cfg = next(c for c in CASES if c.name == "bwd_skew_e64")  # M = H, I multiples of 256
    M.moe_set_gemm_pairs(pairs)
    try:
        ref = _run(cfg)
        assert ref["status"] == 0
        M.moe_set_pipeline_wait_limit(200)
        try:
            got = _run(cfg)
        finally:
            M.moe_set_pipeline_wait_limit(0)
        assert got["status"] & 4, got["status"]  # MOE_DEV_TIMEOUT
        again = _run(cfg)
    finally:
        M.moe_set_gemm_pairs(True)
    assert again["status"] == 0
    for k in ("dx", "dwg", "dbias", "dw13", "dw2"):
        assert torch.equal(again[k].view(torch.uint8), ref[k].view(torch.uint8)), k
