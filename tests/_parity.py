"""Comparison of the CUDA path with the oracle (shared by the GPU tests).

Acceptance rules:
 * logits: the GPU's bf16-rounded routed logits equal the oracle's, except
   where the oracle's exact logit lies within the fp32-accumulation error
   bound of a bf16 rounding midpoint; there the GPU may take the neighbouring
   bf16 value (one step, never more). Bound: 2 * (H + 2) * 2^-24 * sum|x*W|,
   the worst case of any summation order of H+1 terms in fp32 with at most one
   ulp of error per addition.
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


def bf16_neighbours(v: np.ndarray):
    """bf16 values one step below and above each bf16-valued double."""
    f = v.astype(np.float32)
    bits = f.view(np.uint32) >> 16
    up = np.where(f >= 0, bits + 1, bits - 1).astype(np.uint32)
    dn = np.where(f > 0, bits - 1, np.where(f == 0, 0x8001, bits + 1)).astype(np.uint32)
    upv = (up << 16).view(np.float32).astype(np.float64)
    dnv = (dn << 16).view(np.float32).astype(np.float64)
    return dnv, upv


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
            H = ri.H
            delta = 2.0 * (H + 2) * 2.0 ** -24 * ref.absdot
            dn, up = bf16_neighbours(ref.zhat)
            t, e = np.nonzero(diff)
            for a, b in zip(t, e):
                g, zh, z = zg[a, b], ref.zhat[a, b], ref.z[a, b]
                assert g == dn[a, b] or g == up[a, b], (
                    f"row {rows[a]} expert {b}: gpu {g} vs oracle {zh} is more than one bf16 step")
                mid = 0.5 * (g + zh)
                assert abs(z - mid) <= delta[a, b], (
                    f"row {rows[a]} expert {b}: exact logit {z} is {abs(z - mid):.3g} from the "
                    f"rounding midpoint, beyond the accumulation bound {delta[a, b]:.3g}")
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
