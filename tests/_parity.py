"""Comparison of the CUDA path with the oracle (shared by the GPU tests).

Acceptance rules:
 * logits: each GPU bf16 logit must be the bf16 rounding of some value within
   delta of the exact sum z, i.e. lie in [bf16(z - delta), bf16(z + delta)];
   where it differs from the oracle's bf16(z) it is counted. delta is the
   worst-case error of the kernel's fp32 summation tree, one ulp (2^-24
   relative) per addition on the chain, times sum|x*W| (+|bias|), doubled:
     small-M path  : per warp a chain of mma.sync K=16 steps over its share of
                     K, then 8 warps and the K ranges added in a fixed order;
                     bounded by ceil(H/64) + 48 additions
     tcgen05 path  : one fp32 accumulator update per K=16 instruction, so
                     H/16 sequential additions (+32 for the in-instruction sum).
   Near-zero logits (heavy cancellation) can therefore move several bf16
   steps; logits near the top-k are ~1e3 ulps larger and move at most one.
 * selection: the oracle's top-k + softmax applied to the GPU's own logits
   reproduces the GPU's ids exactly and its weights within 2e-6 relative
   (absolute 4 * 2^-149 below the fp32 normal range).
 * agreement: every row whose ids differ from the oracle's has a logit that
   legitimately rounded the other way (counted, reported).
 * on rows without such logits: ids bit-exact, routed weights within 2e-6.
 * shared slot: id E, weight within 2e-6 relative of the oracle's.
 * align: bit-exact against the oracle's align on the GPU's ids.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

import oracle
from moe_router_top_gb300 import inputs

W_RTOL = 2e-6
W_ATOL = 4 * 2.0 ** -149


def weights_close(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.abs(got - ref) <= np.maximum(W_RTOL * np.abs(ref), W_ATOL)


def accumulation_bound(ri: inputs.RouteInputs) -> float:
    """Relative fp32 summation bound (times sum|x*W|) of the kernel path."""
    u = 2.0 ** -24
    if ri.M <= 16:
        chain = -(-ri.H // 64) + 48
    else:
        chain = -(-ri.H // 16) + 32
    return 2.0 * chain * u


@dataclasses.dataclass
class RouteReport:
    rows: int
    logit_mismatch: int = 0          # logits that took the other rounding
    rows_with_mismatch: int = 0
    rows_ids_differ: int = 0         # rows whose ids differ from the oracle's
    max_w_rel: float = 0.0
    max_shared_rel: float = 0.0


def check_route(ri: inputs.RouteInputs, ids_g: np.ndarray, w_g: np.ndarray,
                logits_g: Optional[np.ndarray], rows: Optional[np.ndarray] = None,
                exact_logits: bool = False) -> RouteReport:
    """Compare GPU route outputs (for `rows`, default all) with the oracle."""
    rows = np.arange(ri.M) if rows is None else np.asarray(rows)
    ids_g = np.asarray(ids_g)[rows]
    w_g = np.asarray(w_g)[rows]
    k, S, E = ri.topk, ri.has_shared, ri.E
    ref = oracle.route(ri.x, ri.w, ri.ws, ri.bias, k, ri.shared_scale, rows=rows)
    rep = RouteReport(rows=len(rows))
    row_bad = np.zeros(len(rows), bool)
    if logits_g is not None:
        zg = inputs.bf16_bits_to_f32(np.asarray(logits_g)[rows]).astype(np.float64)
        diff = zg != ref.zhat
        if diff.any():
            assert not exact_logits, f"{int(diff.sum())} logits differ on exact-arithmetic inputs"
            delta = accumulation_bound(ri) * ref.absdot
            t, e = np.nonzero(diff)
            z = ref.z[t, e]
            lo = oracle.bf16_round(z - delta[t, e])
            hi = oracle.bf16_round(z + delta[t, e])
            g = zg[t, e]
            bad = (g < lo) | (g > hi)
            if bad.any():
                j = int(np.argmax(bad))
                raise AssertionError(
                    f"{int(bad.sum())} logits outside the accumulation bound; e.g. row {rows[t[j]]} "
                    f"expert {e[j]}: gpu {g[j]} vs exact {z[j]} (allowed [{lo[j]}, {hi[j]}])")
            rep.logit_mismatch = int(diff.sum())
            row_bad = diff.any(axis=1)
            rep.rows_with_mismatch = int(row_bad.sum())
        # selection on the GPU's own logits must be exact
        sel_ids, sel_w = oracle.select_rows(zg, k)
        assert np.array_equal(ids_g[:, :k], sel_ids), "top-k differs from oracle selection on the GPU's logits"
        ok = weights_close(w_g[:, :k], sel_w)
        assert ok.all(), f"weights off on GPU logits: max rel {np.max(np.abs(w_g[:, :k] - sel_w) / np.maximum(np.abs(sel_w), 1e-30)):.3g}"
    ids_differ = ~np.all(ids_g[:, :k] == ref.ids[:, :k], axis=1)
    rep.rows_ids_differ = int(ids_differ.sum())
    assert not (ids_differ & ~row_bad).any(), (
        f"rows {rows[ids_differ & ~row_bad][:8]} choose different experts without a rounding excuse")
    good = ~row_bad
    if good.any():
        assert np.array_equal(ids_g[good, :k], ref.ids[good, :k])
        ok = weights_close(w_g[good, :k], ref.w[good, :k])
        assert ok.all(), "routed weights beyond 2e-6 relative"
        rel = np.abs(w_g[good, :k].astype(np.float64) - ref.w[good, :k]) / np.maximum(np.abs(ref.w[good, :k]), 1e-30)
        rep.max_w_rel = float(rel.max())
    if S:
        assert np.all(ids_g[:, k] == E), "shared slot id must be E"
        ok = weights_close(w_g[:, k], ref.w[:, k])
        rel = np.abs(w_g[:, k].astype(np.float64) - ref.w[:, k]) / np.maximum(np.abs(ref.w[:, k]), 1e-30)
        rep.max_shared_rel = float(rel.max())
        assert ok.all(), f"shared weight beyond 2e-6 relative (max {rep.max_shared_rel:.3g})"
    return rep


def check_route_properties(ri: inputs.RouteInputs, ids_g: np.ndarray, w_g: np.ndarray) -> None:
    """Invariants that hold at any size, checked on every row."""
    k, S, E = ri.topk, ri.has_shared, ri.E
    routed = np.asarray(ids_g)[:, :k]
    assert routed.min() >= 0 and routed.max() < E
    srt = np.sort(routed, axis=1)
    assert np.all(srt[:, 1:] != srt[:, :-1]), "duplicate expert in a row"
    w = np.asarray(w_g, np.float64)
    assert np.all(np.abs(w[:, :k].sum(axis=1) - 1.0) <= 1e-5), "routed weights do not sum to 1"
    assert np.all(np.diff(w[:, :k], axis=1) <= 0), "routed weights must be non-increasing by slot"
    if S:
        assert np.all(np.asarray(ids_g)[:, k] == E)
        assert np.all((w[:, k] >= 0) & (w[:, k] <= ri.shared_scale))


def check_align(ids_g: np.ndarray, E_al: int, A: int, sorted_g, eids_g, npp_g) -> oracle.AlignResult:
    ref = oracle.align(np.asarray(ids_g), E_al, A)
    npp = int(np.asarray(npp_g).reshape(-1)[0])
    assert npp == ref.npp, f"npp {npp} != oracle {ref.npp}"
    assert np.array_equal(np.asarray(sorted_g)[:npp], ref.sorted_ids), "sorted_token_ids differ"
    assert np.array_equal(np.asarray(eids_g)[: npp // A], ref.expert_ids), "expert_ids differ"
    return ref
