"""The dispatch layout through the entry point that allocates nothing.

moe_dispatch_layout_noalloc serves callers that cannot allocate device memory
when they run (a fully pre-planned memory pool, or a setting where a
cudaMalloc would stall the device or is not allowed): it takes no workspace
and uses a fixed scratch array owned by the library.  These tests call it
through the C ABI and check that it gives exactly the layout of the ordinary
entry point (which uses a caller-allocated workspace), on two calls in a row
with different inputs, so that nothing a call leaves in the shared scratch can
change the next result.  This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _lib():
    from top_routing_dispatch_gb300 import _lib
    return _lib


def _routing(n, E, K, seed, hot=False):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    idx = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(n)]).to(torch.int32)
    if hot:                       # one expert takes half the tokens; some experts stay empty
        idx[: n // 2, 0] = 1
    return idx.cuda()


def _outputs(n, E, K):
    dev = torch.device("cuda:0")
    nK = n * K
    return dict(counts=torch.full((E,), -7, dtype=torch.int32, device=dev),
                offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
                perm=torch.full((nK,), -7, dtype=torch.int32, device=dev),
                inv=torch.full((nK,), -7, dtype=torch.int32, device=dev),
                status=torch.zeros(1, dtype=torch.int32, device=dev))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _run(lib, L, n, E, K, idx, noalloc):
    desc = L.LayerDesc(n, 2048, 1024, E, K, L.MOE_BF16, 0)
    o = _outputs(n, E, K)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if noalloc:
        st = lib.moe_dispatch_layout_noalloc(ctypes.byref(desc), _ptr(idx), _ptr(o["counts"]),
                                             _ptr(o["offsets"]), _ptr(o["perm"]),
                                             _ptr(o["inv"]), _ptr(o["status"]), stream)
    else:
        ws_bytes = lib.moe_layout_workspace_size(ctypes.byref(desc))
        ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda:0")
        st = lib.moe_dispatch_layout(ctypes.byref(desc), _ptr(idx), _ptr(o["counts"]),
                                     _ptr(o["offsets"]), _ptr(o["perm"]), _ptr(o["inv"]),
                                     _ptr(o["status"]), _ptr(ws), ws_bytes, stream)
    assert st == 0, L.STATUS.get(st, st)
    assert lib.moe_check_status(_ptr(o["status"]), stream) == 0
    return {k: v.cpu().numpy() for k, v in o.items()}


@pytest.mark.parametrize("first,second", [
    ((4096, 64, 8, 1, False), (3001, 256, 8, 2, True)),     # large then larger-E, ragged
    ((16384, 64, 8, 3, True), (37, 8, 2, 4, False)),        # large then tiny
])
def test_noalloc_layout_matches_workspace_layout(first, second):
    L = _lib()
    lib = L.load()
    for n, E, K, seed, hot in (first, second):
        idx = _routing(n, E, K, seed, hot)
        ref = _run(lib, L, n, E, K, idx, noalloc=False)
        got = _run(lib, L, n, E, K, idx, noalloc=True)
        for k in ("counts", "offsets", "perm", "inv"):
            assert np.array_equal(got[k], ref[k]), k


def test_noalloc_rejects_layouts_beyond_its_scratch():
    L = _lib()
    lib = L.load()
    K = 8
    n = L.NOALLOC_MAX_PAIRS // K + 1
    desc = L.LayerDesc(n, 2048, 1024, 64, K, L.MOE_BF16, 0)
    nullp = ctypes.c_void_p(None)
    dummy = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    st = lib.moe_dispatch_layout_noalloc(ctypes.byref(desc), _ptr(dummy), _ptr(dummy),
                                         _ptr(dummy), _ptr(dummy), _ptr(dummy), _ptr(dummy),
                                         nullp)
    assert st == 3  # MOE_ERR_WORKSPACE, before anything is enqueued
    # the largest accepted size
    n = L.NOALLOC_MAX_PAIRS // K
    idx = _routing(n, 64, K, 5)
    ref = _run(lib, L, n, 64, K, idx, noalloc=False)
    got = _run(lib, L, n, 64, K, idx, noalloc=True)
    for k in ("counts", "offsets", "perm", "inv"):
        assert np.array_equal(got[k], ref[k]), k
