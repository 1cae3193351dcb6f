"""ctypes loader of the in-tree CUDA library (libmoe_gb300.so).

There is no fallback: if the library has not been built, loading fails loudly.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libmoe_gb300.so")

_lock = threading.Lock()
_lib = None

P, I, U, SZ, LL = C.c_void_p, C.c_int, C.c_uint, C.c_size_t, C.c_longlong

# name -> (restype, argtypes); names and argument order are those of include/moe_gb300.h
SIGNATURES = {
    "moe_route_topk": (I, [P, I, I, I, P, I, P, U, P]),
    "moe_permute_workspace_size": (SZ, [I, I, I]),
    "moe_permute_kernel_launches": (I, [I, I, I]),
    "moe_permute": (I, [P, I, I, P, I, I, I, P, P, P, P, P, P, U, P, SZ, P]),
    "moe_permute_noalloc_max_scratch": (SZ, []),
    "moe_permute_noalloc": (I, [P, I, I, P, I, I, I, P, P, P, P, P, P, U, P]),
    "moe_quant_mxfp8_grouped": (I, [P, I, I, P, I, P, P, U, P]),
    "moe_unpermute_combine": (I, [P, P, P, I, I, I, P, P]),
    "moe_unpermute_combine_backward": (I, [P, P, P, P, I, I, I, P, P, P, P, P]),
    "moe_permute_backward": (I, [P, P, I, I, I, P, P]),
    "moe_route_topk_backward": (I, [P, P, I, P, I, I, I, U, P, P]),
    "moe_route_sigmoid_topk": (I, [P, P, I, I, I, P, I, P, U, P]),
    "moe_amax_bf16": (I, [P, LL, I, P, P, P]),
    "moe_permute_nvfp4": (I, [P, I, I, P, I, I, I, P, P, P, P, P, P, P, P, SZ, P]),
    "moe_quant_nvfp4": (I, [P, LL, I, P, P, P, P, P]),
    "moe_grouped_gemm_up_nvfp4": (I, [P, P, P, P, P, P, P, I, I, I, I, P, P, P, P]),
    "moe_grouped_gemm_down_nvfp4": (I, [P, P, P, P, P, P, P, I, I, I, I, P, P]),
    "moe_route_sigmoid_topk_backward": (I, [P, P, I, P, I, I, I, U, P, P]),
    "moe_packed_weights_bytes": (SZ, [I, I, I, I, I]),
    "moe_prepare_weights": (I, [P, P, P, I, I, I, I, P, P, P, P, P]),
    "moe_grouped_swiglu_gemm": (I, [P, P, P, P, P, P, I, P, I, I, I, I, P, P, P, P]),
    "moe_grouped_gemm_up": (I, [P, P, P, P, I, P, I, I, I, I, P, P, P, P, P]),
    "moe_grouped_gemm_down": (I, [P, P, P, P, I, P, I, I, I, I, P, P]),
    "moe_prepare_weights_bwd": (I, [P, P, P, I, I, I, I, P, P, P, P, P]),
    "moe_grouped_swiglu_dgrad": (I, [P, P, P, P, P, I, P, I, I, I, I, P, P, P, P]),
    "moe_grouped_gemm_dx": (I, [P, P, P, P, I, P, I, I, I, I, P, P]),
    "moe_grouped_transpose_kpad": (SZ, [I, I]),
    "moe_grouped_transpose": (I, [P, P, I, I, P, I, I, P, P, P]),
    "moe_grouped_gemm_wgrad": (I, [P, P, P, P, I, P, I, I, I, I, P, P, P]),
    "moe_get_device_errors": (I, [C.POINTER(C.c_uint32), I]),
    "moe_debug_bounded_wait_selftest": (I, [C.c_uint32, P]),
    "moe_status_string": (C.c_char_p, [I]),
    "moe_route_ids_bytes": (SZ, [I, I, I]),
    "moe_route_probs_bytes": (SZ, [I, I]),
    "moe_ep_recv_expert_ids": (I, [P, I, I, LL, P, P]),
    "moe_host_mapped_pointer": (I, [P, C.POINTER(C.c_void_p)]),
}


class MoeLibraryMissing(RuntimeError):
    pass


def load():
    """Load the library (once) and declare every exported entry point."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise MoeLibraryMissing(
                    f"{LIB_PATH} not found: build the CUDA library first "
                    "(python -m dropless_moe_expert_router_gb300.build)")
            lib = C.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib
