"""The C ABI library builds, loads, exports what include/moe.h declares, and
its host-only calls behave -- no GPU needed (no call here reaches the device)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")

needs_nvcc = pytest.mark.skipif(
    not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")),
    reason="CUDA toolkit not installed")


@pytest.fixture(scope="module")
def lib():
    from top_routing_dispatch_gb300 import build as B
    B.build()
    from top_routing_dispatch_gb300 import _lib
    return _lib.load()


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)


def test_header_matches_binding_list():
    from top_routing_dispatch_gb300 import _lib
    assert sorted(set(header_functions())) == sorted(_lib.SYMBOLS)


@needs_nvcc
def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


@needs_nvcc
def test_exported_dynamic_symbols(lib):
    out = os.popen(f"nm -D --defined-only {lib._name}").read()
    exported = set(re.findall(r"\bT (moe_[a-z0-9_]+)\b", out))
    assert set(header_functions()) <= exported


@needs_nvcc
def test_version_and_status_strings(lib):
    assert b"sm_103a" in lib.moe_version()
    for code in range(8):
        assert lib.moe_status_string(code)
    assert lib.moe_status_string(99) == b"unknown status"


def _desc(**kw):
    from top_routing_dispatch_gb300._lib import LayerDesc
    d = dict(n=4096, H=2048, I=1024, E=64, K=8, dtype=1, norm_topk_prob=0)
    d.update(kw)
    return LayerDesc(**d)


@needs_nvcc
def test_workspace_sizes(lib):
    d = _desc()
    ws = lib.moe_workspace_size(ctypes.byref(d))
    nK = 4096 * 8
    # x_perm + h + y_perm dominate
    assert ws >= nK * 2048 * 2 * 2 + nK * 1024 * 2
    assert ws % 256 == 0
    lw = lib.moe_layout_workspace_size(ctypes.byref(d))
    assert lw == ((nK + 2047) // 2048) * 65 * 4      # one histogram per 2048-pair chunk
    hw = lib.moe_host_workspace_size(ctypes.byref(d))
    assert hw == ws + 4 * 4096 * 2048 * 2             # two staging slots of x and y
    assert lib.moe_workspace_size(ctypes.byref(_desc(E=0))) == 0
    assert lib.moe_host_workspace_size(ctypes.byref(_desc(E=0))) == 0
    assert lib.moe_workspace_size(None) == 0


@needs_nvcc
def test_workspace_slots_are_ordered_and_aligned(lib):
    d = _desc(n=100, H=256, I=128, E=8, K=2)
    base = 1 << 20
    per = lib.moe_workspace_size(ctypes.byref(d))
    prev = None
    for mb in range(2):
        for which in range(11):
            p = lib.moe_workspace_slot(ctypes.byref(d), ctypes.c_void_p(base), mb, which)
            assert p % 256 == 0
            assert base + mb * per <= p < base + (mb + 1) * per
            if prev is not None:
                assert p > prev
            prev = p
    assert lib.moe_workspace_slot(ctypes.byref(d), ctypes.c_void_p(base), 0, 11) is None
    assert lib.moe_workspace_slot(ctypes.byref(d), None, 0, 0) is None


@needs_nvcc
@pytest.mark.parametrize("bad", [
    dict(n=-1), dict(H=0), dict(E=0), dict(K=0), dict(K=9, E=8), dict(dtype=7),
])
def test_invalid_desc_rejected_before_any_launch(lib, bad):
    d = _desc(**bad)
    nullp = ctypes.c_void_p(None)
    st = lib.moe_route_topk(ctypes.byref(d), nullp, nullp, nullp, nullp, nullp, nullp, nullp)
    assert st == 1  # MOE_ERR_INVALID_ARG
    st = lib.moe_permute(ctypes.byref(d), nullp, nullp, nullp, nullp, nullp)
    assert st == 1


@needs_nvcc
@pytest.mark.parametrize("bad,code", [
    (dict(E=300), 2), (dict(K=17, E=64), 2), (dict(H=2047), 2),
])
def test_unsupported_sizes(lib, bad, code):
    d = _desc(**bad)
    nullp = ctypes.c_void_p(None)
    st = lib.moe_combine(ctypes.byref(d), nullp, nullp, nullp, nullp, nullp, nullp)
    assert st == code


@needs_nvcc
def test_gemm_shape_rules(lib):
    nullp = ctypes.c_void_p(None)
    for kw in (dict(I=1000), dict(H=2048 + 32)):   # bf16 needs I % 128, H % 64
        d = _desc(**kw)
        st = lib.moe_grouped_swiglu(ctypes.byref(d), nullp, nullp, nullp, nullp, nullp, nullp, 0,
                                    nullp, nullp)
        assert st == 2
    # null pointers with a valid shape
    st = lib.moe_grouped_swiglu(ctypes.byref(_desc()), nullp, nullp, nullp, nullp, nullp, nullp,
                                0, nullp, nullp)
    assert st == 1


@needs_nvcc
def test_forward_microbatches_argument_checks(lib):
    d = _desc(n=64, H=256, I=128, E=8, K=2)
    nullp = ctypes.c_void_p(None)
    xs = (ctypes.c_void_p * 2)(4096, 8192)
    # misaligned workspace
    st = lib.moe_forward_microbatches(ctypes.byref(d), 2, xs, ctypes.c_void_p(256), nullp,
                                      ctypes.c_void_p(256), ctypes.c_void_p(256), xs,
                                      ctypes.c_void_p(16), 1 << 30, 0, nullp, nullp, nullp)
    assert st == 1
    # too small a workspace
    st = lib.moe_forward_microbatches(ctypes.byref(d), 2, xs, ctypes.c_void_p(256), nullp,
                                      ctypes.c_void_p(256), ctypes.c_void_p(256), xs,
                                      ctypes.c_void_p(1 << 20), 1024, 0, nullp, nullp, nullp)
    assert st == 3
    # bad micro-batch count
    st = lib.moe_forward_microbatches(ctypes.byref(d), 0, xs, ctypes.c_void_p(256), nullp,
                                      ctypes.c_void_p(256), ctypes.c_void_p(256), xs,
                                      ctypes.c_void_p(1 << 20), 1 << 30, 0, nullp, nullp, nullp)
    assert st == 1


@needs_nvcc
def test_forward_host_argument_checks(lib):
    """Checks that return before any CUDA call (no GPU needed)."""
    d = _desc(n=64, H=256, I=128, E=8, K=2)
    nullp = ctypes.c_void_p(None)
    need = lib.moe_host_workspace_size(ctypes.byref(d))
    assert need > 0 and need % 256 == 0
    ws = ctypes.c_void_p(1 << 20)
    fake = ctypes.c_void_p(1 << 12)  # never dereferenced: every call below fails first

    def call(**kw):
        a = dict(x=fake, wg=fake, w13=fake, w2=fake, y=fake, ws=ws, nbytes=need, call=0, dd=d)
        a.update(kw)
        return lib.moe_forward_host(ctypes.byref(a["dd"]), a["x"], a["wg"], nullp, a["w13"],
                                    a["w2"], a["y"], a["ws"], a["nbytes"], a["call"], nullp,
                                    nullp, nullp, nullp)
    assert call(ws=nullp) == 1                                  # MOE_ERR_INVALID_ARG
    assert call(ws=ctypes.c_void_p((1 << 20) + 16)) == 1        # ws not 256-byte aligned
    assert call(call=-1) == 1
    assert call(w13=nullp) == 1
    assert call(nbytes=need - 1) == 3                           # MOE_ERR_WORKSPACE
    assert call(dd=_desc(n=64, H=256, I=100, E=8, K=2)) == 2    # bf16 GEMM needs I % 128
    assert call(dd=_desc(n=64, H=256, I=128, E=8, K=2), x=nullp) == 1


@needs_nvcc
def test_backward_workspace_and_argument_checks(lib):
    """moe_backward_workspace_size is the sum of its 256-byte-aligned slots
    (dY, dw, dh, dG|dU, dx_perm, dlogits, the 16 dW_gate/dbias partials, the
    weight gradients' 16-row tails), and moe_backward rejects bad arguments
    before any CUDA call."""
    up = lambda b: (b + 255) // 256 * 256
    n, H, I, E, K = 4096, 2048, 1024, 64, 8
    nK = n * K
    d = _desc()
    want = sum(up(b) for b in (nK * H * 2, nK * 4, nK * I * 2, nK * 2 * I * 2, nK * H * 2,
                               n * E * 4, 16 * (H + 1) * E * 4, E * 16 * (H + 2 * I) * 2))
    need = lib.moe_backward_workspace_size(ctypes.byref(d))
    assert need == want
    assert lib.moe_backward_workspace_size(ctypes.byref(_desc(E=0))) == 0
    nullp = ctypes.c_void_p(None)
    fake = ctypes.c_void_p(1 << 12)  # never dereferenced: every call below fails first
    ws = ctypes.c_void_p(1 << 20)

    def call(dd=d, x=fake, dy=fake, dx=fake, dw13=fake, wsp=ws, nbytes=need):
        a = [x, fake, fake, fake, dy] + [fake] * 8 + [dx, fake, nullp, dw13, fake]
        return lib.moe_backward(ctypes.byref(dd), *a, wsp, nbytes, nullp, nullp)
    assert call(dd=_desc(dtype=0)) == 2                      # float32 layers: unsupported
    assert call(dd=_desc(H=2112)) == 2                       # H % 256
    assert call(dd=_desc(I=1088)) == 2                       # I % 128
    assert call(x=nullp) == 1
    assert call(dy=nullp) == 1
    assert call(dw13=nullp) == 1
    assert call(wsp=nullp) == 1
    assert call(wsp=ctypes.c_void_p((1 << 20) + 16)) == 1    # ws not 256-byte aligned
    assert call(dx=ctypes.c_void_p((1 << 12) + 8)) == 1      # dx not 16-byte aligned
    assert call(nbytes=need - 1) == 3                        # MOE_ERR_WORKSPACE


@needs_nvcc
def test_pipeline_wait_limit_control(lib):
    # host-only: a negative limit is rejected, 0 (the default) and a positive
    # limit are accepted; no launch happens
    assert lib.moe_set_pipeline_wait_limit(-1) == 1
    assert lib.moe_set_pipeline_wait_limit(1000) == 0
    assert lib.moe_set_pipeline_wait_limit(0) == 0


@needs_nvcc
def test_gemm_tuning_controls(lib):
    # host-only switches, every value accepted (the results are the same
    # either way), and the defaults put back: pairs on, tails per launch
    for v in (0, 1):
        assert lib.moe_set_gemm_pairs(v) == 0
    for v in (-1, 0, 1, 5):
        assert lib.moe_set_gemm_tails(v) == 0
    assert lib.moe_set_gemm_pairs(1) == 0
    assert lib.moe_set_gemm_tails(-1) == 0


@needs_nvcc
def test_tiled_weights_rejected_where_unsupported(lib):
    import top_routing_dispatch_gb300 as M
    # float32 layers and the backward read row-major weights only
    d = M.make_desc(16, 64, 32, 4, 2, "f32", True, tiled=True)
    assert lib.moe_grouped_swiglu(ctypes.byref(d), None, None, None, None, None, None, 0, None,
                                  None) == 2
    d = M.make_desc(16, 256, 128, 8, 2, "bf16", True, tiled=True)
    assert lib.moe_backward(ctypes.byref(d), *([None] * 19), 0, None, None) == 2
    # an unknown layout is an invalid descriptor
    d = M.make_desc(16, 256, 128, 8, 2, "bf16", True)
    d.weight_layout = 7
    assert lib.moe_workspace_size(ctypes.byref(d)) == 0
    # moe_prepare_weights needs bf16 and the GEMM's shape rules
    d = M.make_desc(16, 64, 32, 4, 2, "f32", True)
    assert lib.moe_prepare_weights(ctypes.byref(d), None, None, None, None, None) == 2
    d = M.make_desc(16, 256, 128, 8, 2, "bf16", True)
    assert lib.moe_prepare_weights(ctypes.byref(d), None, None, None, None, None) == 1
    # moe_prepare_router: bf16 only, both pointers required
    assert lib.moe_prepare_router(ctypes.byref(d), None, None, None) == 1
    d = M.make_desc(16, 64, 32, 4, 2, "f32", True)
    assert lib.moe_prepare_router(ctypes.byref(d), None, None, None) == 2
    # the descriptor carries the optional transposed router weight pointer,
    # 16-byte aligned
    assert M.LayerDesc.w_gate_t.offset == 32
    d = M.make_desc(16, 256, 128, 8, 2, "bf16", True)
    d.w_gate_t = 0x1008
    assert lib.moe_workspace_size(ctypes.byref(d)) == 0
    d.w_gate_t = 0x1000
    assert lib.moe_workspace_size(ctypes.byref(d)) > 0
