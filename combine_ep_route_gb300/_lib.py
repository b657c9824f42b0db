"""ctypes declarations of the C-ABI in ``include/ep.h`` (``libep.so``).

Argument marshalling only: every step of dispatch and combine runs in the
library's CUDA kernels. Loading fails loudly when the library has not been
built; there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libep.so")

EP_MAX_W = 64
EP_MAX_E = 1024
EP_MAX_TOPK = 16
EP_MAX_EXTRA = 4

EP_OK = 0
EP_ERR_INVALID_ARG = -1
EP_ERR_CAPACITY = -2
EP_ERR_STATE = -3
EP_ERR_EXPERT_ID = -4
EP_ERR_DUPLICATE = -5
EP_ERR_TIMEOUT = -6
EP_ERR_WORKSPACE = -7
EP_ERR_CUDA = -8
EP_ERR_SCRATCH_LIMIT = -9
EP_STATIC_SCRATCH_BYTES = 4 << 20

EP_BF16 = 1
EP_F32 = 2
EP_FP8 = 3
EP_FP4X2 = 4

EP_PATH_FUSED = 0
EP_PATH_SENDBUF = 1

EP_FLAG_ZERO_PAD = 1
EP_FLAG_SENDBUF = 2
EP_FLAG_WEIGHT_ON_INPUT = 4

EP_OPT_WAIT_LIMIT_NS = 1
EP_OPT_KERNEL_TIMING = 2
EP_OPT_PDL = 3
EP_OPT_MOVE_CTAS_PER_SM = 4
EP_OPT_MOVE_PIPES = 5
EP_OPT_FAULT_SKIP_PUBLISH = 6
EP_OPT_COMBINE_CTAS_PER_SM = 7
EP_OPT_MOVE_CHUNK_BYTES = 8
EP_OPT_MOVE_MAX_STAGES = 9
EP_OPT_FUSED_DISPATCH = 10
EP_OPT_ROUTE_CTAS = 11
EP_OPT_SMALL_DISPATCH = 12

(EP_K_ROUTE, EP_K_MOVE_FUSED, EP_K_PACK, EP_K_EXCHANGE, EP_K_DELIVER, EP_K_COMBINE, EP_K_ZERO_PAD,
 EP_K_COMBINE_TWO_STAGE, EP_K_DISPATCH_FUSED, EP_K_DISPATCH_SMALL) = range(10)
EP_K_COUNT = 10
KERNEL_NAMES = ("route", "move_fused", "pack", "exchange", "deliver", "combine", "zero_pad",
                "combine_two_stage", "dispatch_fused", "dispatch_small")


class EpConfigC(C.Structure):
    _fields_ = [("W", C.c_int32), ("E", C.c_int32), ("top_k", C.c_int32),
                ("max_tokens", C.c_int32), ("hidden", C.c_int32), ("x_dtype", C.c_int32),
                ("n_extra", C.c_int32), ("extra_row_bytes", C.c_int32 * EP_MAX_EXTRA),
                ("flags", C.c_uint32)]


class EpMetadataC(C.Structure):
    _fields_ = [("send_cnt", C.c_void_p), ("pair_row", C.c_void_p), ("pair_w", C.c_void_p),
                ("pair_send", C.c_void_p), ("recv_eloc", C.c_void_p), ("recv_w", C.c_void_p),
                ("recv_row", C.c_void_p), ("send_x", C.c_void_p), ("recv_x", C.c_void_p),
                ("slots_per_token", C.c_int32), ("expert_cap", C.c_int32),
                ("row_bytes", C.c_int32), ("reserved", C.c_int32)]


class EpKernelTimesC(C.Structure):
    _fields_ = [("launches", C.c_int64 * EP_K_COUNT), ("total_ms", C.c_double * EP_K_COUNT),
                ("timed", C.c_int64 * EP_K_COUNT)]


class EpRouteOutputsC(C.Structure):
    _fields_ = [("send_cnt", C.c_void_p), ("pair_row", C.c_void_p), ("pair_w", C.c_void_p),
                ("pair_send", C.c_void_p), ("recv_eloc", C.c_void_p), ("recv_w", C.c_void_p),
                ("recv_row", C.c_void_p), ("expert_num_tokens", C.c_void_p), ("status", C.c_void_p)]


class EpAgrsBuffersC(C.Structure):
    _fields_ = [("x_g", C.c_void_p), ("ids_g", C.c_void_p), ("w_g", C.c_void_p), ("y", C.c_void_p),
                ("status", C.c_void_p)]


# name -> (restype, argtypes); mirrors include/ep.h one to one
SIGNATURES = {
    "ep_capacities": (C.c_int, [C.POINTER(EpConfigC), C.POINTER(C.c_int32), C.POINTER(C.c_int32),
                                C.POINTER(C.c_int32)]),
    "ep_workspace_bytes": (C.c_int, [C.POINTER(EpConfigC), C.POINTER(C.c_size_t)]),
    "ep_ctx_create": (C.c_int, [C.POINTER(EpConfigC), C.c_void_p, C.c_size_t,
                                C.POINTER(C.c_void_p)]),
    "ep_ctx_destroy": (C.c_int, [C.c_void_p]),
    "ep_dispatch": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                              C.POINTER(C.c_void_p), C.c_void_p, C.POINTER(C.c_void_p),
                              C.c_void_p, C.c_int32, C.c_void_p]),
    "ep_combine": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]),
    "ep_combine_two_stage": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]),
    "ep_status": (C.c_int, [C.c_void_p, C.c_void_p]),
    "ep_ctx_reset": (C.c_int, [C.c_void_p]),
    "ep_get_metadata": (C.c_int, [C.c_void_p, C.POINTER(EpMetadataC)]),
    "ep_error_string": (C.c_char_p, [C.c_int]),
    "ep_set_option": (C.c_int, [C.c_void_p, C.c_int32, C.c_int64]),
    "ep_kernel_times": (C.c_int, [C.c_void_p, C.POINTER(EpKernelTimesC)]),
    "ep_route_static": (C.c_int, [C.POINTER(EpConfigC), C.c_void_p, C.c_void_p, C.c_void_p,
                                  C.POINTER(EpRouteOutputsC), C.c_void_p]),
    "ep_agrs": (C.c_int, [C.POINTER(EpConfigC), C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                          C.POINTER(EpAgrsBuffersC), C.c_int32, C.c_void_p, C.c_void_p]),
}

_lib = None


def lib() -> C.CDLL:
    """The loaded library; raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
                "g.build()' or python combine_ep_route_gb300/build.py)")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


class EpError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        msg = lib().ep_error_string(code).decode()
        super().__init__(f"{what}: {msg} ({code})" if what else f"{msg} ({code})")


def check(code: int, what: str = "") -> None:
    if code != EP_OK:
        raise EpError(code, what)
