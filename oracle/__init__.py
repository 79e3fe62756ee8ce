"""ctypes access to the plain C oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the package smoke check
in ``__graft_entry__.py`` and by the CPU-baseline leg of ``bench.py``. The
CUDA library never imports, links or calls anything here, and the oracle
imports nothing from the CUDA side.

Arrays cross as numpy buffers; bf16 tensors are ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (-O2, plain scalar code, IEEE semantics)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB: another build of oracle.c (the pins' mutation test
            # points it at copies with a planted mistake)
            lib = ctypes.CDLL(os.environ.get("ORACLE_LIB") or build())
            P = ctypes.c_void_p
            i32, i64, f32, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double
            lib.oracle_bf16_from_double.argtypes = [f64]
            lib.oracle_bf16_from_double.restype = ctypes.c_uint16
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = f64
            lib.oracle_gate_logits.argtypes = [i32, i32, i32, P, i64, P, P, P, P]
            lib.oracle_gate_logits.restype = None
            lib.oracle_select.argtypes = [i32, i32, i32, P, P, P]
            lib.oracle_select.restype = None
            lib.oracle_shared_weight.argtypes = [f64, f32]
            lib.oracle_shared_weight.restype = f32
            lib.oracle_route.argtypes = [i32, i32, i32, i32, i32, f32, i32, i32, P, i64, P, P, P,
                                         P, P, P, P, P, P]
            lib.oracle_route.restype = None
            lib.oracle_route_threads.argtypes = [i32] + lib.oracle_route.argtypes
            lib.oracle_route_threads.restype = i32
            lib.oracle_bf16_round_array.argtypes = [i64, P, P]
            lib.oracle_bf16_round_array.restype = None
            lib.oracle_select_block_size.argtypes = [i32, i32, i32]
            lib.oracle_select_block_size.restype = i32
            lib.oracle_align_capacity.argtypes = [i64, i32, i32]
            lib.oracle_align_capacity.restype = i64
            lib.oracle_align.argtypes = [P, i64, i32, i32, P, i64, P, i64, P]
            lib.oracle_align.restype = i32
            lib.oracle_align_eplb.argtypes = [P, i64, i32, i32, P, P, i32, i32, i32, P, i64, P, i64, P]
            lib.oracle_align_eplb.restype = i32
            lib.oracle_e4m3_from_double.argtypes = [f64]
            lib.oracle_e4m3_from_double.restype = ctypes.c_uint8
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_double.restype = f64
            lib.oracle_quant_fp8.argtypes = [i32, i32, P, i64, P, P]
            lib.oracle_quant_fp8.restype = None
            lib.oracle_expert_gemm.argtypes = [i64, i32, i32, i32, P, P, i64, P, P, P]
            lib.oracle_expert_gemm.restype = None
            _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# --- scalar helpers -----------------------------------------------------------

def bf16_from_double(v: float) -> int:
    return int(_load().oracle_bf16_from_double(float(v)))


def bf16_to_double(b: int) -> float:
    return float(_load().oracle_bf16_to_double(int(b) & 0xFFFF))


def bf16_round(values: np.ndarray) -> np.ndarray:
    """Round each double to bf16 (RNE), returned as doubles."""
    flat = np.ascontiguousarray(np.asarray(values, dtype=np.float64).ravel())
    out = np.empty_like(flat)
    _load().oracle_bf16_round_array(flat.shape[0], _ptr(flat), _ptr(out))
    return out.reshape(np.shape(values))


# --- route ---------------------------------------------------------------------

def gate_logits(x: np.ndarray, w: np.ndarray, bias: Optional[np.ndarray] = None):
    """fp64 logits z [M,E] and sum|x*W| [M,E] for bf16-bit inputs."""
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    M, H = x.shape
    E = w.shape[0]
    z = np.empty((M, E), dtype=np.float64)
    ad = np.empty((M, E), dtype=np.float64)
    _load().oracle_gate_logits(M, H, E, _ptr(x), H, _ptr(w), _ptr(_c(bias, np.float32)),
                               _ptr(z), _ptr(ad))
    return z, ad


def select(zhat_row: np.ndarray, k: int, renormalize: bool = True):
    """Top-k (value desc, id asc) and softmax weights of one row
    (renormalised over the top-k, or the full softmax's at the top-k)."""
    z = _c(zhat_row, np.float64)
    ids = np.empty(k, dtype=np.int32)
    w = np.empty(k, dtype=np.float32)
    _load().oracle_select(z.shape[0], k, 1 if renormalize else 0, _ptr(z), _ptr(ids), _ptr(w))
    return ids, w


def select_rows(zhat: np.ndarray, k: int, renormalize: bool = True):
    zhat = _c(zhat, np.float64)
    M = zhat.shape[0]
    ids = np.empty((M, k), dtype=np.int32)
    w = np.empty((M, k), dtype=np.float32)
    for t in range(M):
        ids[t], w[t] = select(zhat[t], k, renormalize)
    return ids, w


def shared_weight(s: float, scale: float) -> float:
    return float(_load().oracle_shared_weight(float(s), float(scale)))


class RouteResult:
    def __init__(self, ids, w, zhat, z, absdot, s):
        self.ids, self.w, self.zhat, self.z, self.absdot, self.s = ids, w, zhat, z, absdot, s


def route(x: np.ndarray, w: np.ndarray, ws: Optional[np.ndarray], bias: Optional[np.ndarray],
          topk: int, scale: float = 1.0, rows: Optional[np.ndarray] = None,
          threads: int = 1, renormalize: bool = True, shared_bf16: bool = False) -> RouteResult:
    """Full oracle route. ``rows`` restricts it to a subset of token rows;
    ``threads`` > 1 splits the rows over that many host threads (same
    results, rows are independent). ``renormalize`` and ``shared_bf16``:
    see oracle_route in oracle.c."""
    x = _c(x, np.uint16)
    if rows is not None:
        x = np.ascontiguousarray(x[np.asarray(rows)])
    w = _c(w, np.uint16)
    ws = _c(ws, np.uint16)
    bias = _c(bias, np.float32)
    M, H = x.shape
    E = w.shape[0]
    S = 1 if ws is not None else 0
    width = topk + S
    ids = np.empty((M, width), dtype=np.int32)
    wt = np.empty((M, width), dtype=np.float32)
    zhat = np.empty((M, E), dtype=np.float64)
    z = np.empty((M, E), dtype=np.float64)
    ad = np.empty((M, E), dtype=np.float64)
    s = np.zeros(M, dtype=np.float64)
    args = (M, H, E, topk, S, float(scale), 1 if renormalize else 0, 1 if shared_bf16 else 0,
            _ptr(x), H, _ptr(w), _ptr(ws), _ptr(bias),
            _ptr(ids), _ptr(wt), _ptr(zhat), _ptr(z), _ptr(ad), _ptr(s))
    if threads > 1:
        _load().oracle_route_threads(int(threads), *args)
    else:
        _load().oracle_route(*args)
    return RouteResult(ids, wt, zhat, z, ad, s)


# --- align ---------------------------------------------------------------------

def select_block_size(num_tokens: int, topk: int, num_experts: int) -> int:
    return int(_load().oracle_select_block_size(num_tokens, topk, num_experts))


def align_capacity(numel: int, num_experts: int, A: int) -> int:
    return int(_load().oracle_align_capacity(numel, num_experts, A))


class AlignResult:
    def __init__(self, sorted_ids, expert_ids, npp):
        self.sorted_ids, self.expert_ids, self.npp = sorted_ids, expert_ids, npp


def align(ids: np.ndarray, num_experts: int, A: int) -> AlignResult:
    """Sequential moe_align_block_size. Returns only the defined prefixes."""
    flat = np.ascontiguousarray(np.asarray(ids, dtype=np.int32).ravel())
    numel = flat.shape[0]
    cap = align_capacity(numel, num_experts, A)
    sorted_ids = np.full(max(cap, 1), -7, dtype=np.int32)
    expert_ids = np.full(max((cap + A - 1) // A, 1), -7, dtype=np.int32)
    npp = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_align(_ptr(flat), numel, num_experts, A, _ptr(sorted_ids), cap,
                              _ptr(expert_ids), expert_ids.shape[0], _ptr(npp))
    if rc != 0:
        raise ValueError("oracle_align: id out of range or capacity too small")
    n = int(npp[0])
    return AlignResult(sorted_ids[:n].copy(), expert_ids[: n // A].copy(), n)


def align_eplb(ids: np.ndarray, num_experts: int, eplb_map: np.ndarray, eplb_count: np.ndarray,
               num_physical: int, A: int) -> AlignResult:
    """moe_align_block_size behind the EPLB logical->physical remap (see
    oracle_align_eplb in oracle.c). ids [num_tokens, width]; eplb_map
    [num_experts, max_replicas]; eplb_count [num_experts]."""
    ids = np.asarray(ids, dtype=np.int32)
    width = ids.shape[1] if ids.ndim == 2 else 1
    flat = np.ascontiguousarray(ids.ravel())
    mp = np.ascontiguousarray(eplb_map, dtype=np.int32)
    cnt = np.ascontiguousarray(eplb_count, dtype=np.int32)
    numel = flat.shape[0]
    cap = align_capacity(numel, num_physical, A)
    sorted_ids = np.full(max(cap, 1), -7, dtype=np.int32)
    expert_ids = np.full(max((cap + A - 1) // A, 1), -7, dtype=np.int32)
    npp = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_align_eplb(_ptr(flat), numel, width, num_experts, _ptr(mp), _ptr(cnt),
                                   mp.shape[1], num_physical, A, _ptr(sorted_ids), cap,
                                   _ptr(expert_ids), expert_ids.shape[0], _ptr(npp))
    if rc != 0:
        raise ValueError("oracle_align_eplb: id, replica count or physical id out of range")
    n = int(npp[0])
    return AlignResult(sorted_ids[:n].copy(), expert_ids[: n // A].copy(), n)


# --- hidden states to e4m3 -------------------------------------------------------

def e4m3_from_double(v: float) -> int:
    return int(_load().oracle_e4m3_from_double(float(v)))


def e4m3_to_double(c: int) -> float:
    return float(_load().oracle_e4m3_to_double(int(c) & 0xFF))


def quant_fp8(x: np.ndarray):
    """E4M3 codes [M, H] (uint8) and fp32 block scales [M, H/128] of bf16-bit
    hidden states (see oracle_quant_fp8 in oracle.c)."""
    x = _c(x, np.uint16)
    M, H = x.shape
    q = np.empty((M, H), dtype=np.uint8)
    sc = np.empty((M, H // 128), dtype=np.float32)
    _load().oracle_quant_fp8(M, H, _ptr(x), H, _ptr(q), _ptr(sc))
    return q, sc


# --- consumer expert GEMM -------------------------------------------------------

def expert_gemm(x: np.ndarray, ids: np.ndarray, w: np.ndarray):
    """Exact per-slot expert products out[t*width+s] = x[t] . W[ids[t,s]]^T
    (fp64, [numel, N]) and sum|x*W| of each, for bf16-bit x [T, H], ids
    [T, width] and W [E, N, H]."""
    x = _c(x, np.uint16)
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    w = _c(w, np.uint16)
    T, H = x.shape
    width = ids.shape[1]
    E, N, _ = w.shape
    numel = T * width
    out = np.empty((numel, N), dtype=np.float64)
    ad = np.empty((numel, N), dtype=np.float64)
    _load().oracle_expert_gemm(numel, H, N, width, _ptr(ids), _ptr(x), H, _ptr(w), _ptr(out), _ptr(ad))
    return out, ad
