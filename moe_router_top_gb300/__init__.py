"""GB300-native MoE routing front-end: route (gate GEMM, bf16 logits, top-k,
renormalised softmax, shared slot) and moe_align_block_size.

Python names mirror the C ABI of include/smr.h; this layer only turns torch
tensors into pointers, allocates outputs with torch when the caller does not
pass them, and raises on a non-OK status. The work runs in libsmr.so's CUDA
kernels on the caller's current stream. ``SMR_DISABLE=1`` makes every call
raise :class:`SmrUnsupported`, so a caller can take its own fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

from . import _lib
from ._lib import AlignArgs, ExpertGemmArgs, RouteArgs

__all__ = [
    "SmrError", "SmrUnsupported", "Workspace", "route", "align", "route_align",
    "route_align_static", "expert_gemm",
    "select_block_size", "align_capacity", "route_workspace_size", "align_workspace_size",
    "route_align_workspace_size", "get_device_error", "clear_device_error",
    "get_static_device_error", "clear_static_device_error", "test_force_wait_timeout",
    "last_launch_count", "version",
]

ERR_BAD_ID = 1
ERR_WAIT_TIMEOUT = 2
ERR_BAD_SLOT = 4


class SmrError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


class SmrUnsupported(SmrError):
    """The request is outside the implemented contract; fall back."""


def _status_name(status: int) -> str:
    try:
        return _lib.load().smr_status_string(status).decode()
    except Exception:  # library missing while formatting an error
        return f"status {status}"


def _check(status: int) -> None:
    if status == _lib.SMR_OK:
        return
    msg = _lib.load().smr_last_error().decode()
    if status == _lib.SMR_ERR_UNSUPPORTED:
        raise SmrUnsupported(status, msg)
    raise SmrError(status, msg)


def _disabled() -> None:
    if os.environ.get("SMR_DISABLE", "0") not in ("", "0"):
        raise SmrUnsupported(_lib.SMR_ERR_UNSUPPORTED, "disabled by SMR_DISABLE")


def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Workspace:
    """A zero-initialised device buffer that grows on demand.

    The library leaves a workspace ready for its next call (counters back at
    zero, a call tag that only advances), so a workspace is zeroed once (on
    allocation) and can be reused by later calls and CUDA graph replays.
    Calls sharing one workspace must not overlap on the GPU.
    """

    def __init__(self, nbytes: int = 0, device=None):
        torch = _torch()
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.buf = None
        if nbytes:
            self.ensure(nbytes)

    def ensure(self, nbytes: int):
        torch = _torch()
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=self.device)
        return self.buf

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    @property
    def nbytes(self) -> int:
        return self.buf.numel()


_default_ws = {}


def _workspace(ws, nbytes: int, device):
    if ws is None:
        key = (device.type, device.index)
        ws = _default_ws.get(key)
        if ws is None:
            ws = _default_ws[key] = Workspace(0, device)
    if isinstance(ws, Workspace):
        ws.ensure(nbytes)
        return ws.ptr, ws.nbytes
    return ws.data_ptr(), ws.numel() * ws.element_size()


def _route_args(hidden, gate_w, shared_w, bias, topk, shared_scale, renormalize, ids, wts,
                logits_out, shared_logit_bf16=False, hidden_fp8=None, hidden_scales=None) -> RouteArgs:
    torch = _torch()
    if hidden.dtype != torch.bfloat16 or gate_w.dtype != torch.bfloat16:
        raise TypeError("hidden and gate_w must be bfloat16")
    if hidden.dim() != 2 or hidden.stride(1) != 1:
        raise ValueError("hidden must be 2-D [M, H] with unit stride along H")
    if gate_w.dim() != 2 or not gate_w.is_contiguous():
        raise ValueError("gate_w must be a contiguous [E, H] tensor")
    if shared_w is not None and (shared_w.dtype != torch.bfloat16 or not shared_w.is_contiguous()):
        raise ValueError("shared_w must be a contiguous bfloat16 [1, H] tensor")
    if bias is not None and (bias.dtype != torch.float32 or not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous float32 [E] tensor")
    a = RouteArgs()
    a.M, a.H = hidden.shape
    a.E = gate_w.shape[0]
    if gate_w.shape[1] != a.H:
        raise ValueError("gate_w must be [E, H] with the hidden size of `hidden`")
    a.topk = int(topk)
    a.has_shared = 1 if shared_w is not None else 0
    a.shared_scale = float(shared_scale)
    a.renormalize = 1 if renormalize else 0
    a.hidden = _ptr(hidden)
    a.ld_hidden = hidden.stride(0) if a.M > 1 else a.H
    a.gate_w = _ptr(gate_w)
    a.shared_w = _ptr(shared_w)
    a.bias = _ptr(bias)
    a.topk_ids = _ptr(ids)
    a.topk_weights = _ptr(wts)
    a.logits_out = _ptr(logits_out)
    a.shared_logit_bf16 = 1 if shared_logit_bf16 else 0
    if hidden_fp8 is not None:
        M, H = hidden.shape
        if (hidden_fp8.dtype != torch.uint8 or tuple(hidden_fp8.shape) != (M, H)
                or not hidden_fp8.is_contiguous()):
            raise ValueError("hidden_fp8 must be a contiguous uint8 [M, H] tensor (e4m3 codes)")
        if (hidden_scales is None or hidden_scales.dtype != torch.float32
                or tuple(hidden_scales.shape) != (M, H // 128) or not hidden_scales.is_contiguous()):
            raise ValueError("hidden_scales must be a contiguous float32 [M, H // 128] tensor")
        a.hidden_fp8 = _ptr(hidden_fp8)
        a.hidden_scales = _ptr(hidden_scales)
    return a


def _route_outputs(hidden, topk, has_shared, ids, wts):
    torch = _torch()
    M = hidden.shape[0]
    width = topk + (1 if has_shared else 0)
    if ids is None:
        ids = torch.empty((M, width), dtype=torch.int32, device=hidden.device)
    if wts is None:
        wts = torch.empty((M, width), dtype=torch.float32, device=hidden.device)
    return ids, wts


def route(hidden, gate_w, shared_w=None, bias=None, *, topk: int, shared_scale: float = 1.0,
          renormalize: bool = True, shared_logit_bf16: bool = False, topk_ids=None,
          topk_weights=None, logits_out=None, hidden_fp8=None, hidden_scales=None,
          workspace=None, stream=None) -> Tuple:
    """Route M tokens: returns (topk_ids int32 [M, k+S], topk_weights fp32 [M, k+S]).
    hidden_fp8 (uint8 [M, H]) and hidden_scales (float32 [M, H/128]), when
    given, receive the hidden states as e4m3 codes with one scale per 128
    values, written by the same launch."""
    _disabled()
    lib = _lib.load()
    topk_ids, topk_weights = _route_outputs(hidden, topk, shared_w is not None, topk_ids, topk_weights)
    a = _route_args(hidden, gate_w, shared_w, bias, topk, shared_scale, renormalize, topk_ids,
                    topk_weights, logits_out, shared_logit_bf16, hidden_fp8, hidden_scales)
    need = lib.smr_route_workspace_size(ctypes.byref(a))
    wp, wn = _workspace(workspace, need, hidden.device)
    _check(lib.smr_route(ctypes.byref(a), wp, wn, _stream_ptr(stream)))
    return topk_ids, topk_weights


def _align_args(topk_ids, num_tokens, width, num_experts, block_size, routed_topk,
                routed_experts, sorted_ids, expert_ids, npp, eplb=None) -> AlignArgs:
    a = AlignArgs()
    a.topk_ids = _ptr(topk_ids)
    a.num_tokens = int(num_tokens)
    a.width = int(width)
    a.num_experts = int(num_experts)
    a.routed_topk = int(routed_topk)
    a.routed_experts = int(routed_experts)
    a.block_size = int(block_size)
    a.sorted_token_ids = _ptr(sorted_ids)
    a.sorted_cap = 0 if sorted_ids is None else sorted_ids.numel()
    a.expert_ids = _ptr(expert_ids)
    a.expert_cap = 0 if expert_ids is None else expert_ids.numel()
    a.num_tokens_post_padded = _ptr(npp)
    if eplb is not None:
        emap, ecount, nphys = eplb
        a.eplb_map = _ptr(emap)
        a.eplb_count = _ptr(ecount)
        a.eplb_max_replicas = int(emap.shape[1]) if emap.dim() == 2 else 1
        a.num_physical = int(nphys)
    return a


def _eplb(eplb_map, eplb_count, num_physical):
    """(map, count, num_physical) of an EPLB remap, or None."""
    if eplb_map is None:
        return None
    torch = _torch()
    for t in (eplb_map, eplb_count):
        if t is None or t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError("eplb_map [E_al, R] and eplb_count [E_al] must be contiguous int32 tensors")
    return eplb_map, eplb_count, int(num_physical)


def _align_outputs(device, numel, num_experts, A, sorted_ids, expert_ids, npp):
    torch = _torch()
    cap = align_capacity(numel, num_experts, A)
    if sorted_ids is None:
        sorted_ids = torch.empty(max(cap, 1), dtype=torch.int32, device=device)
    if expert_ids is None:
        expert_ids = torch.empty(max((cap + A - 1) // A, 1), dtype=torch.int32, device=device)
    if npp is None:
        npp = torch.empty(1, dtype=torch.int32, device=device)
    return sorted_ids, expert_ids, npp


def align(topk_ids, num_experts: int, block_size: int = 0, *, routed_topk: int = 0,
          routed_experts: int = 0, sorted_token_ids=None, expert_ids=None,
          num_tokens_post_padded=None, eplb_map=None, eplb_count=None, num_physical: int = 0,
          workspace=None, stream=None) -> Tuple:
    """moe_align_block_size of an int32 [num_tokens, width] id matrix,
    optionally behind an EPLB logical->physical remap (eplb_map [E, R],
    eplb_count [E], num_physical; see smr_align_args in include/smr.h).

    Returns (sorted_token_ids, expert_ids, num_tokens_post_padded); only the
    first npp / npp // A entries of the first two are defined."""
    _disabled()
    torch = _torch()
    lib = _lib.load()
    if topk_ids.dtype != torch.int32 or topk_ids.dim() != 2 or not topk_ids.is_contiguous():
        raise ValueError("topk_ids must be a contiguous int32 [num_tokens, width] tensor")
    T, W = topk_ids.shape
    A = block_size if block_size > 0 else select_block_size(T, routed_topk, routed_experts)
    eplb = _eplb(eplb_map, eplb_count, num_physical)
    outs = _align_outputs(topk_ids.device, T * W, num_physical if eplb else num_experts, A,
                          sorted_token_ids, expert_ids, num_tokens_post_padded)
    a = _align_args(topk_ids, T, W, num_experts, block_size, routed_topk, routed_experts, *outs,
                    eplb=eplb)
    need = lib.smr_align_workspace_size(ctypes.byref(a))
    wp, wn = _workspace(workspace, need, topk_ids.device)
    _check(lib.smr_align(ctypes.byref(a), wp, wn, _stream_ptr(stream)))
    return outs


def route_align(hidden, gate_w, shared_w=None, bias=None, *, topk: int, block_size: int = 0,
                shared_scale: float = 1.0, renormalize: bool = True,
                shared_logit_bf16: bool = False, topk_ids=None, topk_weights=None,
                logits_out=None, sorted_token_ids=None, expert_ids=None,
                num_tokens_post_padded=None, eplb_map=None, eplb_count=None,
                num_physical: int = 0, hidden_fp8=None, hidden_scales=None, workspace=None,
                stream=None) -> Tuple:
    """Route then align (one launch for M <= 16 without an EPLB remap).
    Returns (topk_ids, topk_weights, sorted_token_ids, expert_ids,
    num_tokens_post_padded)."""
    _disabled()
    lib = _lib.load()
    S = 1 if shared_w is not None else 0
    topk_ids, topk_weights = _route_outputs(hidden, topk, S, topk_ids, topk_weights)
    ra = _route_args(hidden, gate_w, shared_w, bias, topk, shared_scale, renormalize, topk_ids,
                     topk_weights, logits_out, shared_logit_bf16, hidden_fp8, hidden_scales)
    M, E = ra.M, ra.E
    A = block_size if block_size > 0 else select_block_size(M, topk, E)
    eplb = _eplb(eplb_map, eplb_count, num_physical)
    outs = _align_outputs(hidden.device, M * (topk + S), num_physical if eplb else E + S, A,
                          sorted_token_ids, expert_ids, num_tokens_post_padded)
    aa = _align_args(topk_ids, M, topk + S, E + S, block_size, topk, E, *outs, eplb=eplb)
    need = lib.smr_route_align_workspace_size(ctypes.byref(ra), ctypes.byref(aa))
    wp, wn = _workspace(workspace, need, hidden.device)
    _check(lib.smr_route_align(ctypes.byref(ra), ctypes.byref(aa), wp, wn, _stream_ptr(stream)))
    return (topk_ids, topk_weights) + tuple(outs)


def route_align_static(hidden, gate_w, shared_w=None, bias=None, *, topk: int,
                       block_size: int = 0, shared_scale: float = 1.0, renormalize: bool = True,
                       shared_logit_bf16: bool = False, topk_ids=None, topk_weights=None,
                       logits_out=None, sorted_token_ids=None, expert_ids=None,
                       num_tokens_post_padded=None, stream=None) -> Tuple:
    """route_align for 1 <= M <= 16 without a workspace: the library's fixed
    device scratch array is used instead, for callers that cannot allocate
    device memory. Calls must not overlap on the GPU; the first call on a
    device must come before any stream capture. Same outputs as route_align.
    (Passing the outputs in avoids the allocations this wrapper otherwise
    makes with torch for convenience.)"""
    _disabled()
    lib = _lib.load()
    S = 1 if shared_w is not None else 0
    topk_ids, topk_weights = _route_outputs(hidden, topk, S, topk_ids, topk_weights)
    ra = _route_args(hidden, gate_w, shared_w, bias, topk, shared_scale, renormalize, topk_ids,
                     topk_weights, logits_out, shared_logit_bf16)
    M, E = ra.M, ra.E
    A = block_size if block_size > 0 else select_block_size(M, topk, E)
    outs = _align_outputs(hidden.device, M * (topk + S), E + S, A, sorted_token_ids, expert_ids,
                          num_tokens_post_padded)
    aa = _align_args(topk_ids, M, topk + S, E + S, block_size, topk, E, *outs)
    _check(lib.smr_route_align_static(ctypes.byref(ra), ctypes.byref(aa), _stream_ptr(stream)))
    return (topk_ids, topk_weights) + tuple(outs)


def expert_gemm(hidden, expert_w, sorted_token_ids, expert_ids, num_tokens_post_padded, *,
                width: int, block_size: int, out=None, workspace=None, stream=None):
    """The consumer expert GEMM over the align's outputs: returns out fp32
    [num_tokens * width, N], row t * width + s = hidden[t] . W[e]^T for the
    slot's expert e (expert_w bf16 [num_experts, N, H]); blocks at or past
    num_tokens_post_padded do no work."""
    _disabled()
    torch = _torch()
    lib = _lib.load()
    if hidden.dtype != torch.bfloat16 or hidden.dim() != 2 or hidden.stride(1) != 1:
        raise ValueError("hidden must be a bfloat16 [T, H] tensor with unit stride along H")
    if expert_w.dtype != torch.bfloat16 or expert_w.dim() != 3 or not expert_w.is_contiguous():
        raise ValueError("expert_w must be a contiguous bfloat16 [num_experts, N, H] tensor")
    T, H = hidden.shape
    E, N, H2 = expert_w.shape
    if H2 != H:
        raise ValueError("expert_w's last dimension must be H")
    if out is None:
        out = torch.empty((T * width, N), dtype=torch.float32, device=hidden.device)
    a = ExpertGemmArgs()
    a.hidden, a.ld_hidden = _ptr(hidden), (hidden.stride(0) if T > 1 else H)
    a.num_tokens, a.width, a.H = T, int(width), H
    a.expert_w, a.num_experts, a.N = _ptr(expert_w), E, N
    a.block_size = int(block_size)
    a.sorted_token_ids, a.sorted_cap = _ptr(sorted_token_ids), sorted_token_ids.numel()
    a.expert_ids, a.num_tokens_post_padded = _ptr(expert_ids), _ptr(num_tokens_post_padded)
    a.out = _ptr(out)
    wp, wn = _workspace(workspace, 256, hidden.device)
    _check(lib.smr_expert_gemm(ctypes.byref(a), wp, wn, _stream_ptr(stream)))
    return out


def select_block_size(num_tokens: int, topk: int, num_experts: int) -> int:
    return int(_lib.load().smr_select_block_size(num_tokens, topk, num_experts))


def align_capacity(numel: int, num_experts: int, block_size: int) -> int:
    return int(_lib.load().smr_align_capacity(numel, num_experts, block_size))


def route_workspace_size(args: RouteArgs) -> int:
    return int(_lib.load().smr_route_workspace_size(ctypes.byref(args)))


def align_workspace_size(args: AlignArgs) -> int:
    return int(_lib.load().smr_align_workspace_size(ctypes.byref(args)))


def route_align_workspace_size(route_args: RouteArgs, align_args: AlignArgs) -> int:
    return int(_lib.load().smr_route_align_workspace_size(ctypes.byref(route_args),
                                                          ctypes.byref(align_args)))


def get_device_error(workspace, stream=None) -> int:
    """Sticky error bits of a workspace (synchronises the stream)."""
    lib = _lib.load()
    ptr = workspace.ptr if isinstance(workspace, Workspace) else workspace.data_ptr()
    code = ctypes.c_int32(0)
    _check(lib.smr_get_device_error(ptr, _stream_ptr(stream), ctypes.byref(code)))
    return code.value


def clear_device_error(workspace, stream=None) -> None:
    lib = _lib.load()
    ptr = workspace.ptr if isinstance(workspace, Workspace) else workspace.data_ptr()
    _check(lib.smr_clear_device_error(ptr, _stream_ptr(stream)))


def get_static_device_error(stream=None) -> int:
    """Sticky error bits of route_align_static's fixed scratch array on the
    current device (synchronises the stream)."""
    code = ctypes.c_int32(0)
    _check(_lib.load().smr_get_static_device_error(_stream_ptr(stream), ctypes.byref(code)))
    return code.value


def clear_static_device_error(stream=None) -> None:
    _check(_lib.load().smr_clear_static_device_error(_stream_ptr(stream)))


STALL_NONE = _lib.SMR_STALL_NONE
STALL_SMALL_TAIL = _lib.SMR_STALL_SMALL_TAIL
STALL_TC_MERGE = _lib.SMR_STALL_TC_MERGE


def test_force_wait_timeout(site: int, limit: int = 1) -> None:
    """Test hook: make one bounded wait of later launches run out (see
    smr_test_force_wait_timeout in include/smr.h); STALL_NONE switches it off."""
    _check(_lib.load().smr_test_force_wait_timeout(int(site), int(limit)))


def last_launch_count() -> int:
    return int(_lib.load().smr_last_launch_count())


def version() -> int:
    return int(_lib.load().smr_version())
