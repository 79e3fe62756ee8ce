"""ctypes declarations of the C ABI in include/smr.h (libsmr.so).

Argument marshalling only: every step of the routing path runs in the CUDA
kernels behind these symbols. There is no CPU fallback; if the shared
library is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsmr.so")

SMR_OK = 0
SMR_ERR_INVALID_ARG = 1
SMR_ERR_UNSUPPORTED = 2
SMR_ERR_WORKSPACE = 3
SMR_ERR_CUDA = 4
SMR_ERR_DEVICE = 5

# Every function include/smr.h declares.
EXPORTED = (
    "smr_select_block_size", "smr_align_capacity", "smr_route_workspace_size",
    "smr_align_workspace_size", "smr_route_align_workspace_size", "smr_route", "smr_align",
    "smr_route_align", "smr_get_device_error", "smr_clear_device_error", "smr_status_string",
    "smr_last_error", "smr_version", "smr_last_launch_count", "smr_route_align_static",
    "smr_get_static_device_error", "smr_clear_static_device_error", "smr_test_force_wait_timeout",
    "smr_expert_gemm",
)

SMR_STALL_NONE = 0
SMR_STALL_SMALL_TAIL = 1
SMR_STALL_TC_MERGE = 2


class RouteArgs(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
        ("topk", ctypes.c_int32), ("has_shared", ctypes.c_int32),
        ("shared_scale", ctypes.c_float), ("renormalize", ctypes.c_int32),
        ("hidden", ctypes.c_void_p), ("ld_hidden", ctypes.c_int64),
        ("gate_w", ctypes.c_void_p), ("shared_w", ctypes.c_void_p),
        ("bias", ctypes.c_void_p), ("topk_ids", ctypes.c_void_p),
        ("topk_weights", ctypes.c_void_p), ("logits_out", ctypes.c_void_p),
        ("shared_logit_bf16", ctypes.c_int32),
        ("hidden_fp8", ctypes.c_void_p), ("hidden_scales", ctypes.c_void_p),
    ]


class AlignArgs(ctypes.Structure):
    _fields_ = [
        ("topk_ids", ctypes.c_void_p), ("num_tokens", ctypes.c_int32),
        ("width", ctypes.c_int32), ("num_experts", ctypes.c_int32),
        ("routed_topk", ctypes.c_int32), ("routed_experts", ctypes.c_int32),
        ("block_size", ctypes.c_int32), ("sorted_token_ids", ctypes.c_void_p),
        ("sorted_cap", ctypes.c_int64), ("expert_ids", ctypes.c_void_p),
        ("expert_cap", ctypes.c_int64), ("num_tokens_post_padded", ctypes.c_void_p),
        ("eplb_map", ctypes.c_void_p), ("eplb_count", ctypes.c_void_p),
        ("eplb_max_replicas", ctypes.c_int32), ("num_physical", ctypes.c_int32),
    ]


class ExpertGemmArgs(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_void_p), ("ld_hidden", ctypes.c_int64),
        ("num_tokens", ctypes.c_int32), ("width", ctypes.c_int32), ("H", ctypes.c_int32),
        ("expert_w", ctypes.c_void_p), ("num_experts", ctypes.c_int32), ("N", ctypes.c_int32),
        ("block_size", ctypes.c_int32), ("sorted_token_ids", ctypes.c_void_p),
        ("sorted_cap", ctypes.c_int64), ("expert_ids", ctypes.c_void_p),
        ("num_tokens_post_padded", ctypes.c_void_p), ("out", ctypes.c_void_p),
    ]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libsmr.so and declare its signatures (raises if it is not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        RA, AA = ctypes.POINTER(RouteArgs), ctypes.POINTER(AlignArgs)
        sigs = {
            "smr_select_block_size": ([i32, i32, i32], i32),
            "smr_align_capacity": ([i64, i32, i32], i64),
            "smr_route_workspace_size": ([RA], sz),
            "smr_align_workspace_size": ([AA], sz),
            "smr_route_align_workspace_size": ([RA, AA], sz),
            "smr_route": ([RA, P, sz, P], ctypes.c_int),
            "smr_align": ([AA, P, sz, P], ctypes.c_int),
            "smr_route_align": ([RA, AA, P, sz, P], ctypes.c_int),
            "smr_get_device_error": ([P, P, ctypes.POINTER(i32)], ctypes.c_int),
            "smr_clear_device_error": ([P, P], ctypes.c_int),
            "smr_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "smr_last_error": ([], ctypes.c_char_p),
            "smr_version": ([], i32),
            "smr_last_launch_count": ([], i32),
            "smr_route_align_static": ([RA, AA, P], ctypes.c_int),
            "smr_get_static_device_error": ([P, ctypes.POINTER(i32)], ctypes.c_int),
            "smr_clear_static_device_error": ([P], ctypes.c_int),
            "smr_test_force_wait_timeout": ([i32, i64], ctypes.c_int),
            "smr_expert_gemm": ([ctypes.POINTER(ExpertGemmArgs), P, sz, P], ctypes.c_int),
        }
        for name, (argtypes, restype) in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = argtypes
            fn.restype = restype
        _lib = lib
        return lib
