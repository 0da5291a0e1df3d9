"""Python face of the C ABI: the same calls, taking torch tensors.

torch provides device memory and streams only; every step of the layer runs
in the library's CUDA kernels.  Each function checks the returned status and
raises MoEError on anything but MOE_OK.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import LayerDesc, MOE_BF16, MOE_F32, SLOT  # noqa: F401

_DT = {torch.float32: MOE_F32, torch.bfloat16: MOE_BF16}
_TORCH = {MOE_F32: torch.float32, MOE_BF16: torch.bfloat16}


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        lib = _lib.load()
        msg = lib.moe_status_string(status).decode()
        super().__init__(f"{where}: {_lib.STATUS.get(status, status)} ({msg})")


def _check(status: int, where: str):
    if status != 0:
        raise MoEError(status, where)


def _p(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(s):
    if s is None:
        s = torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream if hasattr(s, "cuda_stream") else int(s))


def make_desc(n, H, I, E, K, dtype, norm_topk_prob, tiled=False, w_gate_t=None) -> LayerDesc:
    """tiled: the expert weights passed to the expert entry points are the
    output of moe_prepare_weights (MOE_WEIGHTS_TILED).  w_gate_t: the router
    weight transposed by moe_prepare_router (the caller keeps the tensor
    alive while the descriptor is used), or None."""
    if isinstance(dtype, torch.dtype):
        dtype = _DT[dtype]
    elif isinstance(dtype, str):
        dtype = {"f32": MOE_F32, "bf16": MOE_BF16}[dtype]
    return LayerDesc(int(n), int(H), int(I), int(E), int(K), int(dtype), int(bool(norm_topk_prob)),
                     int(bool(tiled)), _p(w_gate_t))


def desc_for(cfg, n=None, tiled=False, w_gate_t=None) -> LayerDesc:
    """LayerDesc of a workload config (anything with n, H, I, E, K, dtype, norm_topk_prob)."""
    return make_desc(cfg.n if n is None else n, cfg.H, cfg.I, cfg.E, cfg.K, cfg.dtype,
                     cfg.norm_topk_prob, tiled, w_gate_t)


def moe_prepare_weights(desc, w13, w2, w13_tiled=None, w2_tiled=None, stream=None):
    """w13 and w2 regrouped into contiguous 64 x 64 tiles (MOE_WEIGHTS_TILED);
    returns (w13_tiled, w2_tiled), allocated here when not given."""
    w13_tiled = torch.empty_like(w13) if w13_tiled is None else w13_tiled
    w2_tiled = torch.empty_like(w2) if w2_tiled is None else w2_tiled
    _check(_lib.load().moe_prepare_weights(ctypes.byref(desc), _p(w13), _p(w2), _p(w13_tiled),
                                           _p(w2_tiled), _stream(stream)), "moe_prepare_weights")
    return w13_tiled, w2_tiled


def moe_prepare_router(desc, w_gate, w_gate_t=None, stream=None):
    """w_gate (H, E) transposed into (E, H) for LayerDesc.w_gate_t; returns it
    (allocated here when not given)."""
    H, E = w_gate.shape
    if w_gate_t is None:
        w_gate_t = torch.empty((E, H), dtype=w_gate.dtype, device=w_gate.device)
    _check(_lib.load().moe_prepare_router(ctypes.byref(desc), _p(w_gate), _p(w_gate_t),
                                          _stream(stream)), "moe_prepare_router")
    return w_gate_t


def torch_dtype(desc: LayerDesc):
    return _TORCH[desc.dtype]


# ------------------------------------------------------------ the six calls
def moe_route_topk(desc, x, w_gate, bias, topk_idx, topk_w, logits, stream=None):
    _check(_lib.load().moe_route_topk(ctypes.byref(desc), _p(x), _p(w_gate), _p(bias),
                                      _p(topk_idx), _p(topk_w), _p(logits), _stream(stream)),
           "moe_route_topk")


def moe_layout_workspace_size(desc) -> int:
    return int(_lib.load().moe_layout_workspace_size(ctypes.byref(desc)))


def moe_dispatch_layout(desc, topk_idx, counts, offsets, perm, inv_perm, status_word, ws,
                        stream=None):
    nbytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(_lib.load().moe_dispatch_layout(ctypes.byref(desc), _p(topk_idx), _p(counts),
                                           _p(offsets), _p(perm), _p(inv_perm), _p(status_word),
                                           _p(ws), nbytes, _stream(stream)),
           "moe_dispatch_layout")


def moe_dispatch_layout_noalloc(desc, topk_idx, counts, offsets, perm, inv_perm, status_word,
                                stream=None):
    """moe_dispatch_layout using the library's own fixed scratch array (for
    callers that cannot allocate device memory when they run)."""
    _check(_lib.load().moe_dispatch_layout_noalloc(ctypes.byref(desc), _p(topk_idx), _p(counts),
                                                   _p(offsets), _p(perm), _p(inv_perm),
                                                   _p(status_word), _stream(stream)),
           "moe_dispatch_layout_noalloc")


def moe_permute(desc, x, perm, x_perm, status_word=None, stream=None):
    _check(_lib.load().moe_permute(ctypes.byref(desc), _p(x), _p(perm), _p(x_perm),
                                   _p(status_word), _stream(stream)), "moe_permute")


def moe_permute_scatter(desc, x, inv_perm, x_perm, status_word=None, stream=None):
    """x_perm[inv_perm[t*K + k]] = x[t]: the permute with each x row read once."""
    _check(_lib.load().moe_permute_scatter(ctypes.byref(desc), _p(x), _p(inv_perm), _p(x_perm),
                                           _p(status_word), _stream(stream)),
           "moe_permute_scatter")


def moe_grouped_swiglu(desc, x_perm, w13, w2, offsets, h, y_perm, sm_reserve=0, status_word=None,
                       stream=None):
    _check(_lib.load().moe_grouped_swiglu(ctypes.byref(desc), _p(x_perm), _p(w13), _p(w2),
                                          _p(offsets), _p(h), _p(y_perm), int(sm_reserve),
                                          _p(status_word), _stream(stream)),
           "moe_grouped_swiglu")


def moe_expert_gemm1_swiglu(desc, x_perm, w13, offsets, h, sm_reserve=0, status_word=None,
                            stream=None):
    _check(_lib.load().moe_expert_gemm1_swiglu(ctypes.byref(desc), _p(x_perm), _p(w13),
                                               _p(offsets), _p(h), int(sm_reserve),
                                               _p(status_word), _stream(stream)),
           "moe_expert_gemm1_swiglu")


def moe_expert_gemm1_swiglu_gather(desc, x, perm, w13, offsets, h, sm_reserve=0,
                                   status_word=None, stream=None):
    _check(_lib.load().moe_expert_gemm1_swiglu_gather(
        ctypes.byref(desc), _p(x), _p(perm), _p(w13), _p(offsets), _p(h), int(sm_reserve),
        _p(status_word), _stream(stream)), "moe_expert_gemm1_swiglu_gather")


def moe_expert_gemm2(desc, h, w2, offsets, y_perm, sm_reserve=0, status_word=None, stream=None):
    _check(_lib.load().moe_expert_gemm2(ctypes.byref(desc), _p(h), _p(w2), _p(offsets),
                                        _p(y_perm), int(sm_reserve), _p(status_word),
                                        _stream(stream)), "moe_expert_gemm2")


def moe_expert_gemm2_weighted(desc, h, w2, offsets, perm, topk_w, y_slot, sm_reserve=0,
                              status_word=None, stream=None):
    _check(_lib.load().moe_expert_gemm2_weighted(
        ctypes.byref(desc), _p(h), _p(w2), _p(offsets), _p(perm), _p(topk_w), _p(y_slot),
        int(sm_reserve), _p(status_word), _stream(stream)), "moe_expert_gemm2_weighted")


def moe_combine_slots(desc, y_slot, y, stream=None):
    _check(_lib.load().moe_combine_slots(ctypes.byref(desc), _p(y_slot), _p(y), _stream(stream)),
           "moe_combine_slots")


def moe_combine(desc, y_perm, topk_w, inv_perm, y, status_word=None, stream=None):
    _check(_lib.load().moe_combine(ctypes.byref(desc), _p(y_perm), _p(topk_w), _p(inv_perm),
                                   _p(y), _p(status_word), _stream(stream)), "moe_combine")


def kernels_per_forward(desc) -> int:
    """Kernel launches one micro-batch of moe_forward_microbatches enqueues."""
    return int(_lib.load().moe_forward_launches(ctypes.byref(desc)))


def moe_workspace_size(desc) -> int:
    return int(_lib.load().moe_workspace_size(ctypes.byref(desc)))


def moe_forward_microbatches(desc, xs, w_gate, bias, w13, w2, ys, ws, sm_reserve=0,
                             status_word=None, compute=None, dispatch=None):
    n = len(xs)
    xa = (ctypes.c_void_p * n)(*[x.data_ptr() for x in xs])
    ya = (ctypes.c_void_p * n)(*[y.data_ptr() for y in ys])
    nbytes = ws.numel() * ws.element_size()
    _check(_lib.load().moe_forward_microbatches(
        ctypes.byref(desc), n, xa, _p(w_gate), _p(bias), _p(w13), _p(w2), ya, _p(ws), nbytes,
        int(sm_reserve), _p(status_word), _stream(compute),
        _stream(dispatch) if dispatch is not None else ctypes.c_void_p(None)),
        "moe_forward_microbatches")


def moe_host_workspace_size(desc) -> int:
    return int(_lib.load().moe_host_workspace_size(ctypes.byref(desc)))


def moe_forward_host(desc, x_host, w_gate, bias, w13, w2, y_host, ws, call, status_word=None,
                     compute=None, copy_in=None, copy_out=None):
    nbytes = ws.numel() * ws.element_size()
    opt = lambda s: _stream(s) if s is not None else ctypes.c_void_p(None)
    _check(_lib.load().moe_forward_host(
        ctypes.byref(desc), _p(x_host), _p(w_gate), _p(bias), _p(w13), _p(w2), _p(y_host),
        _p(ws), nbytes, int(call), _p(status_word), _stream(compute), opt(copy_in),
        opt(copy_out)), "moe_forward_host")


def moe_workspace_slot(desc, ws, mb, which) -> int:
    if isinstance(which, str):
        which = SLOT[which]
    p = _lib.load().moe_workspace_slot(ctypes.byref(desc), _p(ws), int(mb), int(which))
    if not p:
        raise ValueError("bad workspace slot request")
    return int(p)


def moe_set_pipeline_wait_limit(cycles):
    """Test control: cycles a tensor-core GEMM pipeline wait waits before it
    gives up with MOE_ERR_TIMEOUT (0: the default, about a second)."""
    _check(_lib.load().moe_set_pipeline_wait_limit(int(cycles)), "moe_set_pipeline_wait_limit")


def moe_set_gemm_pairs(enable):
    """Tuning control: run the tensor-core grouped GEMMs (forward and
    backward) on CTA pairs (True, the default) or on single CTAs (False); the
    results are bitwise the same."""
    _check(_lib.load().moe_set_gemm_pairs(1 if enable else 0), "moe_set_gemm_pairs")


def moe_set_gemm_tails(mode):
    """Tuning control of the forward pair GEMMs' fused tails: None (the
    default) chooses per launch, False never, True always; the results are
    bitwise the same."""
    m = -1 if mode is None else (1 if mode else 0)
    _check(_lib.load().moe_set_gemm_tails(m), "moe_set_gemm_tails")


def moe_check_status(status_word, stream=None) -> int:
    """Synchronises `stream` and returns the mapped status code (0 = OK)."""
    return int(_lib.load().moe_check_status(_p(status_word), _stream(stream)))


# ------------------------------------------------------------ conveniences
def workspace_view(desc, ws, mb, name):
    """A torch view of one micro-batch's intermediate inside the workspace."""
    dt = torch_dtype(desc)
    nK = desc.n * desc.K
    shapes = dict(logits=((desc.n, desc.E), torch.float32), topk_idx=((desc.n, desc.K), torch.int32),
                  topk_w=((desc.n, desc.K), torch.float32), counts=((desc.E,), torch.int32),
                  offsets=((desc.E + 1,), torch.int32), perm=((nK,), torch.int32),
                  inv_perm=((nK,), torch.int32), x_perm=((nK, desc.H), dt), h=((nK, desc.I), dt),
                  y_perm=((nK, desc.H), dt), status=((1,), torch.int32))
    shape, dtype = shapes[name]
    addr = moe_workspace_slot(desc, ws, mb, name)
    base = ws.data_ptr()
    off = addr - base
    esz = torch.empty((), dtype=dtype).element_size()
    count = 1
    for s in shape:
        count *= s
    flat = ws.view(torch.uint8)[off:off + count * esz].view(dtype)
    return flat.view(*shape)


class MoELayer:
    """One MoE expert layer with resident weights and a reusable workspace.

    weights: w_gate (H,E), w13 (E,H,2I), w2 (E,I,H) in the layer dtype on the
    device, bias (E,) float32 or None.
    """

    def __init__(self, desc: LayerDesc, w_gate, bias, w13, w2, num_mb=1, w_gate_t=None):
        """w_gate_t: the router weight transposed (moe_prepare_router), kept
        alive here and set in this layer's copy of the descriptor."""
        if w_gate_t is not None:
            desc = LayerDesc.from_buffer_copy(desc)
            desc.w_gate_t = w_gate_t.data_ptr()
        self.desc = desc
        self.w_gate, self.bias, self.w13, self.w2 = w_gate, bias, w13, w2
        self.w_gate_t = w_gate_t
        dev = w13.device
        self.num_mb = num_mb
        self.ws = torch.empty(moe_workspace_size(desc) * num_mb, dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def forward(self, xs, ys=None, sm_reserve=0, compute=None, dispatch=None):
        if ys is None:
            ys = [torch.empty_like(x) for x in xs]
        moe_forward_microbatches(self.desc, xs, self.w_gate, self.bias, self.w13, self.w2, ys,
                                 self.ws, sm_reserve, self.status, compute, dispatch)
        return ys

    def __call__(self, x):
        return self.forward([x])[0]

    def view(self, name, mb=0):
        return workspace_view(self.desc, self.ws, mb, name)

    def check(self, stream=None):
        _check(moe_check_status(self.status, stream), "device status")


def moe_backward_workspace_size(desc) -> int:
    """Bytes of device scratch moe_backward needs for this layer shape."""
    return int(_lib.load().moe_backward_workspace_size(ctypes.byref(desc)))


def moe_backward(desc, x, w_gate, w13, w2, dy, logits, topk_idx, topk_w, offsets, inv_perm,
                 x_perm, h, y_perm, dx, dw_gate, dbias, dw13, dw2, ws, status_word=None,
                 stream=None):
    """Gradients of the layer for dy (bf16 layers): dx (n,H) bf16 and the
    float32 dw_gate (H,E), dbias (E, or None), dw13 (E,H,2I), dw2 (E,I,H),
    from the forward's own intermediates (logits, topk_idx, topk_w, offsets,
    inv_perm, x_perm, h and the unweighted y_perm of moe_expert_gemm2)."""
    nbytes = ws.numel() * ws.element_size()
    _check(_lib.load().moe_backward(
        ctypes.byref(desc), _p(x), _p(w_gate), _p(w13), _p(w2), _p(dy), _p(logits), _p(topk_idx),
        _p(topk_w), _p(offsets), _p(inv_perm), _p(x_perm), _p(h), _p(y_perm), _p(dx),
        _p(dw_gate), _p(dbias), _p(dw13), _p(dw2), _p(ws), nbytes, _p(status_word),
        _stream(stream)), "moe_backward")


class HostPipeline:
    """moe_forward_host over one staging workspace: each call enqueues the copy
    of a pinned host x in, the layer, and the copy of y out, on three streams,
    so consecutive calls overlap their copies with their neighbours' layers.
    y_host of a call is final after `synchronize()` (or once an event recorded
    on `copy_out` after the call has completed)."""

    def __init__(self, layer: MoELayer, compute=None, copy_in=None, copy_out=None):
        dev = layer.w13.device
        self.layer = layer
        self.ws = torch.empty(moe_host_workspace_size(layer.desc), dtype=torch.uint8, device=dev)
        self.compute = compute if compute is not None else torch.cuda.current_stream(dev)
        self.copy_in = copy_in if copy_in is not None else torch.cuda.Stream(device=dev)
        self.copy_out = copy_out if copy_out is not None else torch.cuda.Stream(device=dev)
        self.calls = 0

    def __call__(self, x_host, y_host):
        L = self.layer
        moe_forward_host(L.desc, x_host, L.w_gate, L.bias, L.w13, L.w2, y_host, self.ws,
                         self.calls, L.status, self.compute, self.copy_in, self.copy_out)
        self.calls += 1
        return y_host

    def synchronize(self):
        self.copy_out.synchronize()
