"""ctypes binding of include/moe.h and include/lm_head.h (same names; argument
marshalling only).

Every step of the layer runs in the CUDA library ``_build/libwse.so``.  There
is no Python or CPU fallback: if the library is missing or fails to load,
``lib()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build_lib

_lock = threading.Lock()
_lib = None

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_OOM = 4
MOE_ERR_DEVICE_TIMEOUT = 5
MOE_MAX_TOKENS = 64
MOE_LM_HEAD_MAX_TOKENS = 16
MOE_GEMV_MAX_TOKENS = 16
MOE_GEMV_CUDA_CORES = 0
MOE_GEMV_TENSOR_CORES = 1
MOE_FWD_NO_PDL = 0x1
MOE_FWD_GRAPH = 0x2
MOE_FWD_TRACE = 0x4
MOE_FWD_OUT_F32 = 0x8
MOE_FWD_TEST_SKIP_ARRIVAL = 0x40000000
TRACE_SLOTS = 32

STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
                4: "MOE_ERR_OOM", 5: "MOE_ERR_DEVICE_TIMEOUT"}


class moe_info_t(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_experts", ctypes.c_int), ("topk", ctypes.c_int),
                ("inter", ctypes.c_int), ("max_tokens", ctypes.c_int), ("n_sms", ctypes.c_int),
                ("gateup_stages", ctypes.c_int), ("down_stages", ctypes.c_int),
                ("gateup_tile_bytes", ctypes.c_int), ("down_tile_bytes", ctypes.c_int),
                ("weight_bytes", ctypes.c_size_t), ("workspace_bytes", ctypes.c_size_t),
                ("kernels_per_forward", ctypes.c_int), ("router_split", ctypes.c_int),
                ("smem_bytes", ctypes.c_size_t), ("shared_expert", ctypes.c_int),
                ("routed_scale", ctypes.c_float), ("bias_selection_only", ctypes.c_int),
                ("fp8_experts", ctypes.c_int), ("grid_ctas", ctypes.c_int),
                ("wait_limit_ns", ctypes.c_ulonglong)]


class moe_layer_opts_t(ctypes.Structure):
    _fields_ = [("w_shared_gate_up", ctypes.c_void_p), ("w_shared_down", ctypes.c_void_p),
                ("routed_scale", ctypes.c_float), ("bias_selection_only", ctypes.c_int)]


class MoEError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def library_path() -> str:
    return build_lib.LIB


def lib(build_if_missing: bool = True):
    """The loaded C library with its prototypes declared."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = build_lib.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"CUDA library not built: {path}")
            build_lib.build()
        L = ctypes.CDLL(path)
        vp, ci, cu = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint
        i32p = ctypes.POINTER(ctypes.c_int32)
        f32p = ctypes.POINTER(ctypes.c_float)
        ip = ctypes.POINTER(ctypes.c_int)
        L.moe_create.argtypes = [ci, ci, ci, ci, vp, vp, vp]
        L.moe_create.restype = vp
        L.moe_create_ex.argtypes = [ci, ci, ci, ci, vp, vp, vp, ctypes.POINTER(moe_layer_opts_t)]
        L.moe_create_ex.restype = vp
        L.moe_create_fp8.argtypes = [ci, ci, ci, ci, vp, vp, vp, vp, vp]
        L.moe_create_fp8.restype = vp
        L.moe_forward.argtypes = [vp, vp, vp, vp, ci, vp]
        L.moe_forward.restype = ci
        L.moe_forward_ex.argtypes = [vp, vp, vp, vp, vp, ci, vp, cu]
        L.moe_forward_ex.restype = ci
        L.moe_forward_timed.argtypes = [vp, vp, vp, vp, ci, vp, ctypes.POINTER(vp)]
        L.moe_forward_timed.restype = ci
        L.moe_set_router_bias.argtypes = [vp, vp]
        L.moe_set_router_bias.restype = ci
        L.moe_get_status.argtypes = [vp]
        L.moe_get_status.restype = ci
        L.moe_set_grid.argtypes = [vp, ci]
        L.moe_set_grid.restype = ci
        L.moe_set_wait_limit.argtypes = [vp, ctypes.c_ulonglong]
        L.moe_set_wait_limit.restype = ci
        L.moe_combine_partials.argtypes = [vp, ci, ctypes.c_size_t, vp, vp]
        L.moe_combine_partials.restype = ci
        L.moe_get_info.argtypes = [vp, ctypes.POINTER(moe_info_t)]
        L.moe_get_info.restype = ci
        L.moe_read_routing.argtypes = [vp, ci, ip, ip, i32p, i32p, i32p, i32p, f32p, ci]
        L.moe_read_routing.restype = ci
        L.moe_read_trace.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64), ci]
        L.moe_read_trace.restype = ci
        L.moe_route_static.argtypes = [ci, ci, ci, vp, vp, vp, ci, vp, vp, vp]
        L.moe_route_static.restype = ci
        L.moe_route_static_read_status.argtypes = [vp, vp]
        L.moe_route_static_read_status.restype = ci
        L.moe_destroy.argtypes = [vp]
        L.moe_destroy.restype = None
        L.moe_lm_head_create.argtypes = [ci, ci, vp]
        L.moe_lm_head_create.restype = vp
        L.moe_lm_head_forward.argtypes = [vp, vp, vp, ci, vp]
        L.moe_lm_head_forward.restype = ci
        L.moe_lm_head_get_status.argtypes = [vp]
        L.moe_lm_head_get_status.restype = ci
        L.moe_lm_head_destroy.argtypes = [vp]
        L.moe_lm_head_destroy.restype = None
        L.moe_gemv_pack.argtypes = [vp, vp, ci, ci, vp]
        L.moe_gemv_pack.restype = ci
        L.moe_gemv.argtypes = [vp, vp, vp, ci, ci, ci, ci, vp]
        L.moe_gemv.restype = ci
        L.moe_gemv_get_status.argtypes = []
        L.moe_gemv_get_status.restype = ci
        L.moe_last_error.argtypes = []
        L.moe_last_error.restype = ctypes.c_char_p
        _lib = L
        return L


def last_error() -> str:
    return (lib().moe_last_error() or b"").decode()


def check(fn: str, status: int):
    if status != MOE_OK:
        raise MoEError(fn, status, last_error())
