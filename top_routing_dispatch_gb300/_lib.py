"""ctypes binding of libmoe_gb300.so (the C ABI declared in include/moe.h).

Argument marshalling only.  Loading fails loudly if the library has not been
built: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

LIB_NAME = "libmoe_gb300.so"
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), LIB_NAME)

# C ABI symbols, in header order (tests check the library exports each one).
SYMBOLS = (
    "moe_version", "moe_status_string", "moe_route_topk", "moe_layout_workspace_size",
    "moe_dispatch_layout", "moe_dispatch_layout_noalloc", "moe_permute", "moe_permute_scatter", "moe_grouped_swiglu", "moe_expert_gemm1_swiglu",
    "moe_expert_gemm1_swiglu_gather", "moe_expert_gemm2", "moe_combine",
    "moe_workspace_size", "moe_forward_launches", "moe_forward_microbatches", "moe_workspace_slot", "moe_check_status",
    "moe_host_workspace_size", "moe_forward_host", "moe_expert_gemm2_weighted",
    "moe_combine_slots", "moe_backward_workspace_size", "moe_backward",
    "moe_set_pipeline_wait_limit", "moe_prepare_weights", "moe_set_gemm_pairs",
    "moe_prepare_router", "moe_set_gemm_tails",
)

MOE_F32, MOE_BF16 = 0, 1
MOE_WEIGHTS_ROW_MAJOR, MOE_WEIGHTS_TILED = 0, 1
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_BAD_ROUTING", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_TIMEOUT",
          7: "MOE_ERR_BAD_LAYOUT"}
DEV_BAD_ROUTING, DEV_BAD_LAYOUT, DEV_TIMEOUT = 0x1, 0x2, 0x4
NOALLOC_MAX_PAIRS = 524288  # MOE_NOALLOC_MAX_PAIRS

# workspace slots of moe_workspace_slot
SLOT = dict(logits=0, topk_idx=1, topk_w=2, counts=3, offsets=4, perm=5, inv_perm=6,
            x_perm=7, h=8, y_perm=9, status=10)


class LayerDesc(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("K", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("norm_topk_prob", ctypes.c_int32), ("weight_layout", ctypes.c_int32),
                ("w_gate_t", ctypes.c_void_p)]


_vp = ctypes.c_void_p
_desc_p = ctypes.POINTER(LayerDesc)
_st = ctypes.c_int


def _declare(lib):
    sig = {
        "moe_version": (ctypes.c_char_p, []),
        "moe_forward_launches": (ctypes.c_int, [_desc_p]),
        "moe_status_string": (ctypes.c_char_p, [_st]),
        "moe_route_topk": (_st, [_desc_p, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
        "moe_layout_workspace_size": (ctypes.c_size_t, [_desc_p]),
        "moe_dispatch_layout": (_st, [_desc_p, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                      ctypes.c_size_t, _vp]),
        "moe_dispatch_layout_noalloc": (_st, [_desc_p, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
        "moe_permute": (_st, [_desc_p, _vp, _vp, _vp, _vp, _vp]),
        "moe_permute_scatter": (_st, [_desc_p, _vp, _vp, _vp, _vp, _vp]),
        "moe_grouped_swiglu": (_st, [_desc_p, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int,
                                     _vp, _vp]),
        "moe_expert_gemm1_swiglu": (_st, [_desc_p, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, _vp]),
        "moe_expert_gemm1_swiglu_gather": (_st, [_desc_p, _vp, _vp, _vp, _vp, _vp, ctypes.c_int,
                                                 _vp, _vp]),
        "moe_expert_gemm2": (_st, [_desc_p, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, _vp]),
        "moe_combine": (_st, [_desc_p, _vp, _vp, _vp, _vp, _vp, _vp]),
        "moe_workspace_size": (ctypes.c_size_t, [_desc_p]),
        "moe_forward_microbatches": (_st, [_desc_p, ctypes.c_int, ctypes.POINTER(_vp), _vp, _vp,
                                           _vp, _vp, ctypes.POINTER(_vp), _vp, ctypes.c_size_t,
                                           ctypes.c_int, _vp, _vp, _vp]),
        "moe_workspace_slot": (_vp, [_desc_p, _vp, ctypes.c_int, ctypes.c_int]),
        "moe_check_status": (_st, [_vp, _vp]),
        "moe_set_pipeline_wait_limit": (_st, [ctypes.c_longlong]),
        "moe_set_gemm_pairs": (_st, [ctypes.c_int]),
        "moe_set_gemm_tails": (_st, [ctypes.c_int]),
        "moe_prepare_weights": (_st, [_desc_p, _vp, _vp, _vp, _vp, _vp]),
        "moe_prepare_router": (_st, [_desc_p, _vp, _vp, _vp]),
        "moe_host_workspace_size": (ctypes.c_size_t, [_desc_p]),
        "moe_expert_gemm2_weighted": (_st, [_desc_p, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int,
                                            _vp, _vp]),
        "moe_combine_slots": (_st, [_desc_p, _vp, _vp, _vp]),
        "moe_backward_workspace_size": (ctypes.c_size_t, [_desc_p]),
        "moe_backward": (_st, [_desc_p] + [_vp] * 19 + [ctypes.c_size_t, _vp, _vp]),
        "moe_forward_host": (_st, [_desc_p, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t,
                                   ctypes.c_longlong, _vp, _vp, _vp, _vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_LIB = None


def load():
    """The loaded library (cached).  Raises ImportError when it is missing."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing; build it with `python -m top_routing_dispatch_gb300.build`")
        _LIB = _declare(ctypes.CDLL(LIB_PATH))
    return _LIB
