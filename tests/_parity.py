"""Comparison of the CUDA path with the oracle (shared by the GPU tests).

Every quantity that excuses a row is computed from the oracle alone (its
exact logits z, their bf16 roundings zhat and sum|x*W|), never from the GPU's
output. Acceptance rules, per token row:

 * admissible logits: the kernel accumulates in fp32, so its bf16 logit of
   (t, e) may be any bf16 rounding of a value within delta of the exact sum z,
   i.e. lie in [bf16(z - delta), bf16(z + delta)]. delta is the worst-case
   error of the kernel's fp32 summation tree, one ulp (2^-24 relative) per
   addition on the chain, times sum|x*W| (+|bias|), doubled:
     small-M path  : per warp a chain of mma.sync K=16 steps over its share of
                     K, then 8 warps and the K ranges added in a fixed order;
                     bounded by ceil(H/64) + 48 additions
     tcgen05 path  : one fp32 accumulator update per K=16 instruction, so
                     H/16 sequential additions (+32 for the in-instruction sum).
   Only a z within delta of a bf16 rounding boundary has two admissible
   values; far from one both ends round alike.
 * exact row: ids bit-exact against the oracle's and routed weights within
   2e-6 relative (absolute 4 * 2^-149 below the fp32 normal range).
 * rounding row: not exact, but reproduced exactly (ids, and weights within
   2e-6) by the oracle's own selection on an admissible choice of logits:
   with logits_out, the GPU's logits themselves (each must be admissible);
   without, a search over the admissible values of the logits that can reach
   the top-k. The count is reported and bounded by MAX_ROUNDING_FRACTION.
   Without renormalisation (weights = the E-expert softmax at the top-k) a
   flip of ANY logit moves the denominator, so without logits_out such rows
   are held to a weight bound derived from the bands instead (the oracle's
   softmax shares times each band's exponential width); with logits_out the
   check stays exact.
 * boundary row (the benchmark spec): the oracle's k-th and (k+1)-th rounded logits
   tie or lie within 1 bf16 ulp. The expert SET chosen may differ from the
   oracle's only on boundary rows (counted and reported).
 * near-midpoint row (reported): a logit the oracle selects has two
   admissible values, so the GPU's weights may legitimately differ.
 * shared slot: id E, weight within 2e-6 relative of the oracle's.
 * align: bit-exact against the oracle's align on the GPU's ids.
"""
from __future__ import annotations

import dataclasses
import itertools
import os
from typing import List, Optional

import numpy as np

import oracle
from moe_router_top_gb300 import inputs

W_RTOL = 2e-6
W_ATOL = 4 * 2.0 ** -149
# Rows explained only by a legitimate rounding flip, at most this fraction of
# the rows compared (plus MIN_ROUNDING_ROWS, so tiny batches are not held to
# a fraction of one row). Expected: well under 1% on the random workloads.
MAX_ROUNDING_FRACTION = 0.02
MIN_ROUNDING_ROWS = 2
MAX_COMBOS = 1 << 14
MAX_STEPS = 4


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


# --- bf16 neighbours (bit patterns; -0 and +0 are one value) ----------------

def _bits(v: float) -> int:
    return int(np.array([v], np.float32).view(np.uint32)[0] >> 16)


def _val(b: int) -> float:
    return float(np.array([b << 16], np.uint32).view(np.float32)[0])


def bf16_next_down(v: float) -> float:
    """The largest bf16 value below the bf16 value v."""
    if v == 0.0:
        return -_val(0x0001)
    b = _bits(v)
    return _val(b - 1) if v > 0 else _val(b + 1)


def bf16_next_up(v: float) -> float:
    if v == 0.0:
        return _val(0x0001)
    b = _bits(v)
    return _val(b + 1) if v > 0 else (0.0 if b == 0x8001 else _val(b - 1))


def bf16_values_near(v: float, lo: float, hi: float, steps: int) -> List[float]:
    """The bf16 values of [lo, hi] other than v, at most `steps` bf16 steps
    from v, nearest first."""
    out, up, down = [], v, v
    for _ in range(steps):
        up, down = bf16_next_up(up), bf16_next_down(down)
        out += [u for u in (up, down) if lo <= u <= hi]
    return out


@dataclasses.dataclass
class RouteReport:
    rows: int
    exact_rows: int = 0
    rounding_rows: int = 0           # not exact, explained by an admissible rounding
    boundary_rows: int = 0           # oracle: k-th and (k+1)-th tie or within 1 ulp
    near_midpoint_rows: int = 0      # oracle: a selected logit has two admissible values
    set_differs_rows: int = 0        # GPU expert set != oracle's (boundary rows only)
    logit_mismatch: int = 0          # logits_out path: GPU logits != oracle's rounding
    max_w_rel: float = 0.0           # on exact rows
    max_shared_rel: float = 0.0

    def as_dict(self):
        return dataclasses.asdict(self)


def _explained(zhat_row, lo_row, hi_row, k, ids_row, w_row, oracle_ids, renorm=True) -> bool:
    """Does the oracle's selection on some admissible choice of this row's
    logits reproduce (ids_row, w_row)? Only the logits of experts that either
    selection holds can make a difference (any other expert stays out of the
    GPU's top-k at the oracle's value). Each of those may take an admissible
    value up to MAX_STEPS bf16 steps from the oracle's rounding, or from the
    value the GPU's weights imply for it; the choices are tried by the number
    of logits changed (one, then two, ...), at most MAX_COMBOS selections in
    all. An explanation found is admissible by construction (every value lies
    in its band), so the limits only bound the search."""
    cand = sorted(set(ids_row.tolist()) | set(oracle_ids.tolist()))
    others = {}
    for e in cand:
        vals = []
        # where a logit sums terms that nearly cancel, its admissible band
        # spans many bf16 steps; the GPU's weights then imply its value: for
        # e in slot j and another expert r in slot i, w_j / w_i =
        # exp(z_e - z_r), with z_r taken at the oracle's rounding
        if renorm and e in ids_row.tolist() and len(ids_row) > 1:
            j = ids_row.tolist().index(e)
            i = 1 if j == 0 else 0
            if w_row[j] > 0 and w_row[i] > 0:
                implied = float(oracle.bf16_round(np.array(
                    [zhat_row[ids_row[i]] + np.log(float(w_row[j]) / float(w_row[i]))]))[0])
                vals += [implied] + bf16_values_near(implied, lo_row[e], hi_row[e], MAX_STEPS)
        vals += bf16_values_near(zhat_row[e], lo_row[e], hi_row[e], MAX_STEPS)
        seen = set()
        others[e] = [v for v in vals if lo_row[e] <= v <= hi_row[e] and v != zhat_row[e]
                     and not (v in seen or seen.add(v))]
    amb = [e for e in cand if others[e]]
    tried = 0
    z = zhat_row.copy()
    for r in range(1, len(amb) + 1):
        for subset in itertools.combinations(amb, r):
            for combo in itertools.product(*(others[e] for e in subset)):
                tried += 1
                if tried > MAX_COMBOS:
                    return False
                z[list(subset)] = combo
                sid, sw = oracle.select(z, k, renorm)
                z[list(subset)] = zhat_row[list(subset)]
                if np.array_equal(sid, ids_row) and weights_close(w_row, sw).all():
                    return True
    return False


def check_route(ri: inputs.RouteInputs, ids_g: np.ndarray, w_g: np.ndarray,
                logits_g: Optional[np.ndarray] = None, rows: Optional[np.ndarray] = None,
                exact_logits: bool = False, threads: Optional[int] = None) -> RouteReport:
    """Compare GPU route outputs (for `rows`, default all) with the oracle
    under the rules above; returns the counts."""
    rows = np.arange(ri.M) if rows is None else np.asarray(rows)
    ids_g = np.asarray(ids_g)[rows]
    w_g = np.asarray(w_g)[rows]
    k, S, E = ri.topk, ri.has_shared, ri.E
    if threads is None:
        threads = min(os.cpu_count() or 1, 32) if len(rows) >= 256 else 1
    renorm = ri.renormalize
    ref = oracle.route(ri.x, ri.w, ri.ws, ri.bias, k, ri.shared_scale, rows=rows, threads=threads,
                       renormalize=renorm, shared_bf16=ri.shared_bf16)
    n = len(rows)
    rep = RouteReport(rows=n)

    # admissible logits, from the oracle alone
    delta = accumulation_bound(ri) * ref.absdot
    lo = oracle.bf16_round(ref.z - delta)
    hi = oracle.bf16_round(ref.z + delta)
    assert np.all(lo <= ref.zhat) and np.all(ref.zhat <= hi)
    order = np.argsort(-ref.zhat, axis=1, kind="stable")
    sel = order[:, :k]
    near_mid = np.take_along_axis(lo != hi, sel, axis=1).any(axis=1)
    rep.near_midpoint_rows = int(near_mid.sum())
    boundary = np.zeros(n, bool)
    if k < E:
        zk = np.take_along_axis(ref.zhat, order[:, k - 1:k], axis=1)[:, 0]
        zk1 = np.take_along_axis(ref.zhat, order[:, k:k + 1], axis=1)[:, 0]
        down = np.array([bf16_next_down(v) for v in zk])
        boundary = zk1 >= down
    rep.boundary_rows = int(boundary.sum())

    if logits_g is not None:
        zg = inputs.bf16_bits_to_f32(np.asarray(logits_g)[rows]).astype(np.float64)
        zg = zg + 0.0  # -0 and +0 are one value
        bad = (zg < lo) | (zg > hi)
        if bad.any():
            t, e = np.nonzero(bad)
            raise AssertionError(
                f"{int(bad.sum())} logits outside the accumulation bound; e.g. row {rows[t[0]]} "
                f"expert {e[0]}: gpu {zg[t[0], e[0]]} vs exact {ref.z[t[0], e[0]]} "
                f"(allowed [{lo[t[0], e[0]]}, {hi[t[0], e[0]]}])")
        rep.logit_mismatch = int((zg != ref.zhat).sum())
        if exact_logits:
            assert rep.logit_mismatch == 0, f"{rep.logit_mismatch} logits differ on exact-arithmetic inputs"
        # the GPU's selection on its own (admissible) logits must be the
        # oracle's selection on them
        sel_ids, sel_w = oracle.select_rows(zg, k, renorm)
        assert np.array_equal(ids_g[:, :k], sel_ids), "top-k differs from oracle selection on the GPU's logits"
        ok = weights_close(w_g[:, :k], sel_w)
        assert ok.all(), f"weights off on GPU logits: max rel {np.max(np.abs(w_g[:, :k] - sel_w) / np.maximum(np.abs(sel_w), 1e-30)):.3g}"

    same_ids = np.all(ids_g[:, :k] == ref.ids[:, :k], axis=1)
    exact = same_ids & weights_close(w_g[:, :k], ref.w[:, :k]).all(axis=1)
    rep.exact_rows = int(exact.sum())
    if exact_logits:
        assert exact.all(), f"rows {rows[~exact][:8]} differ from the oracle on exact-arithmetic inputs"
    set_differs = np.array([set(ids_g[i, :k].tolist()) != set(ref.ids[i, :k].tolist()) for i in range(n)],
                           dtype=bool)
    rep.set_differs_rows = int(set_differs.sum())
    assert not (set_differs & ~boundary).any(), (
        f"rows {rows[set_differs & ~boundary][:8]} choose other experts than the oracle off the "
        f"k-th boundary")
    if logits_g is None and not renorm and (~exact).any():
        # without renormalisation every logit enters the denominator, so a
        # legitimate rounding flip anywhere in the row moves the weights: each
        # weight may differ relatively by its own logit's band plus the
        # denominator's, sum over e of p_e * (exp(hi_e - lo_e) - 1), p the
        # oracle's softmax (plus the 2e-6 of the arithmetic, and 10%)
        zmax = ref.zhat.max(axis=1, keepdims=True)
        pe = np.exp(ref.zhat - zmax)
        pe /= pe.sum(axis=1, keepdims=True)
        band = np.expm1(hi - lo)
        den_var = (pe * band).sum(axis=1)
        num_var = np.take_along_axis(band, ids_g[:, :k].astype(np.int64), axis=1)
        allowed = 1.1 * (W_RTOL + num_var + den_var[:, None]) * np.abs(ref.w[:, :k]) + W_ATOL
        same_set_rows = ~exact & same_ids
        off = np.abs(w_g[:, :k].astype(np.float64) - ref.w[:, :k]) > allowed
        assert not (off & same_set_rows[:, None]).any(), (
            f"rows {rows[(off & same_set_rows[:, None]).any(axis=1)][:8]}: weights beyond the "
            f"rounding bound of the unrenormalised softmax")
    for i in np.nonzero(~exact)[0]:
        if logits_g is None and renorm:  # with logits_out the GPU's own logits explained it above
            assert _explained(ref.zhat[i], lo[i], hi[i], k, ids_g[i, :k], w_g[i, :k], ref.ids[i, :k],
                              renorm), (
                f"row {rows[i]}: ids {ids_g[i, :k]} / weights differ from the oracle's "
                f"{ref.ids[i, :k]} and no admissible rounding of its logits explains them")
    rep.rounding_rows = int((~exact).sum())
    assert not renorm or rep.rounding_rows <= max(MIN_ROUNDING_ROWS, int(np.ceil(MAX_ROUNDING_FRACTION * n))), (
        f"{rep.rounding_rows} of {n} rows differ by a rounding flip, above the "
        f"{MAX_ROUNDING_FRACTION:.0%} ceiling")
    if exact.any():
        rel = (np.abs(w_g[exact, :k].astype(np.float64) - ref.w[exact, :k]) /
               np.maximum(np.abs(ref.w[exact, :k]), 1e-30))
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
    if ri.renormalize:
        assert np.all(np.abs(w[:, :k].sum(axis=1) - 1.0) <= 1e-5), "routed weights do not sum to 1"
    else:
        assert np.all(w[:, :k].sum(axis=1) <= 1.0 + 1e-5), "routed weights sum above 1"
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


def record(name: str, rep: RouteReport, **extra) -> None:
    """Append a parity report line to $SMR_PARITY_LOG (JSON lines), if set."""
    path = os.environ.get("SMR_PARITY_LOG")
    if not path:
        return
    import json
    with open(path, "a") as f:
        f.write(json.dumps({"case": name, **rep.as_dict(), **extra}) + "\n")
