"""ctypes binding of the C ABI declared in ``include/moe.h``.

Only argument marshalling lives here: every step of the routed branch runs in
the sm_103a kernels of ``libmoe_gb300.so``.  There is no CPU fallback: if the
library cannot be built or loaded, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

c_int, c_size_t, c_void_p, c_char_p = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_char_p
c_int64 = ctypes.c_int64

# name -> (restype, argtypes), mirroring include/moe.h
SIGNATURES = {
    "moe_abi_version": (c_int, []),
    "moe_selftest_bounded_wait": (c_int, [c_void_p, c_void_p]),
    "moe_status_string": (c_char_p, [c_int]),
    "moe_dispatch_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "moe_dispatch": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                             c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_dispatch_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                     c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "moe_dispatch_quant": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                   c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_size_t, c_void_p]),
    "moe_dispatch_quant_ex": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int, c_int,
                                      c_int, c_int, c_int64, c_void_p, c_void_p, c_void_p,
                                      c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_dispatch_source_slots": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int, c_int,
                                          c_int, c_int, c_int, c_void_p, c_void_p, c_void_p,
                                          c_void_p, c_void_p, c_void_p, c_void_p]),
    "moe_expert_compute_source_slots": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                                c_int, c_int, c_void_p, c_void_p, c_void_p,
                                                c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                                c_int, c_void_p]),
    "moe_dispatch_quant_source_slots": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int,
                                                c_int, c_int, c_int, c_int, c_void_p, c_void_p,
                                                c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                                c_void_p]),
    "moe_gemm_source_slots": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                      c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                      c_void_p, c_void_p, c_size_t, c_int, c_void_p]),
    "moe_expert_compute_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int]),
    "moe_expert_compute": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_void_p,
                                   c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_size_t, c_void_p]),
    "moe_combine": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                            c_void_p, c_void_p]),
    "moe_quantize_fp8": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p,
                                 c_void_p]),
    "moe_gemm_gateup_silu": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "moe_gemm_down": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_void_p,
                              c_void_p, c_void_p, c_void_p, c_void_p]),
    "moe_dispatch_packed": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                    c_int, c_int64, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_size_t, c_void_p]),
    "moe_expert_compute_packed_workspace_size": (c_size_t, [c_int64, c_int, c_int]),
    "moe_expert_compute_packed": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int64, c_int, c_int,
                                          c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                          c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_combine_packed": (c_int, [c_void_p, c_int64, c_void_p, c_void_p, c_int, c_int, c_int,
                                   c_void_p, c_void_p]),
    "moe_dispatch_ex": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int, c_int, c_int,
                                c_int, c_int64, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                c_size_t, c_void_p]),
    "moe_expert_compute_ex_workspace_size": (c_size_t, [c_int, c_int, c_int64, c_int, c_int]),
    "moe_expert_compute_ex": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int64, c_int, c_int,
                                      c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                      c_void_p, c_size_t, c_int, c_void_p]),
    "moe_layer_stats": (c_int, [c_void_p, c_int, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                c_void_p, c_void_p, c_void_p]),
    "moe_expert_compute_gemm_launches": (c_int, [c_int, c_int, c_int64, c_int, c_int]),
    "moe_ep_pack_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int]),
    "moe_ep_pack": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_void_p,
                            c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                            c_void_p]),
    "moe_ep_offsets_workspace_size": (c_size_t, [c_int64]),
    "moe_ep_route_offsets": (c_int, [c_void_p, c_int64, c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_ep_return": (c_int, [c_void_p, c_int64, c_void_p, c_void_p, c_void_p, c_int64, c_int, c_int,
                              c_void_p, c_void_p, c_void_p]),
    "moe_ep_result_map": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int, c_int,
                                  c_void_p, c_void_p]),
    "moe_expert_compute_workspace_layout": (c_int, [c_int, c_int, c_int64, c_int, c_int, c_void_p]),
    "moe_gemm_gateup_down_sync_size": (c_size_t, [c_int, c_int, c_int64]),
    "moe_gemm_gateup_down": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int64, c_int,
                                     c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_int,
                                     c_void_p]),
}
W13_INTERLEAVED = 1
GEMM_ONE_LAUNCH = 2
GEMM_TWO_LAUNCHES = 4

STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED",
          -3: "MOE_ERR_WORKSPACE", -4: "MOE_ERR_CUDA"}
DEV_BAD_EXPERT_ID, DEV_CAPACITY_DROPPED, DEV_TIMEOUT = 1, 2, 4

_lock = threading.Lock()
_lib = None


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")
        self.status = status


def load(build_if_stale: bool = True) -> ctypes.CDLL:
    """Load (building first if the sources are newer) the library and declare
    every entry point.  Raises if it cannot."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build() if build_if_stale else _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is missing; run token_dispatch_grouped_topk_gb300.build")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def check(fn: str, status: int) -> None:
    if status != 0:
        raise MoeError(fn, status)
