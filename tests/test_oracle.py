"""Pins for the CPU oracle, against things other than the oracle itself:
brute force on tiny inputs (exact rational arithmetic), library routines on
special cases (torch's fp32->bf16 conversion, numpy matmul, scipy softmax and
expit), closed forms, hand-worked tie cases, invariants, and the numbers the
alignment page prints. CPU only.
"""
from __future__ import annotations

import bisect
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

import oracle
from moe_router_top_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# --------------------------------------------------------------- bf16 pins ---

def _bf16_table():
    """All finite bf16 values except -0, as (Fraction, bits), sorted by value."""
    table = []
    for b in range(0x10000):
        exp = (b >> 7) & 0xFF
        if exp == 0xFF or b == 0x8000:
            continue
        frac = b & 0x7F
        if exp == 0:
            mag = Fraction(frac, 1 << 7) * Fraction(1, 1 << 126)
        else:
            mag = (1 + Fraction(frac, 1 << 7)) * (Fraction(2) ** (exp - 127))
        table.append((-mag if b & 0x8000 else mag, b))
    table.sort()
    return table


_TABLE = None


def _brute_bf16(v: float) -> int:
    """Nearest bf16 by exhaustive table search; ties to the even bit pattern."""
    global _TABLE
    if _TABLE is None:
        _TABLE = _bf16_table()
    if v == 0.0:
        return 0x8000 if math.copysign(1.0, v) < 0 else 0x0000
    x = Fraction(v)
    keys = [t[0] for t in _TABLE]
    vmax = keys[-1]
    half_ulp_max = Fraction(2) ** (127 - 8)
    if abs(x) >= vmax + half_ulp_max:
        return 0xFF80 if x < 0 else 0x7F80
    i = bisect.bisect_left(keys, x)
    cands = [_TABLE[j] for j in (i - 1, i) if 0 <= j < len(_TABLE)]
    best = min(cands, key=lambda t: (abs(t[0] - x), t[1] & 1))
    if best[0] == 0:  # rounds to zero: keep the sign of x
        return 0x8000 if x < 0 else 0x0000
    return best[1]


@pytest.mark.parametrize("v,bits", [
    (1.0, 0x3F80), (-2.0, 0xC000), (0.0, 0x0000), (-0.0, 0x8000),
    (257.0, 0x4380),            # 257 is a midpoint -> even neighbour 256
    (259.0, 0x4382),            # 259 is a midpoint -> even neighbour 260
    (258.0, 0x4381),            # exactly representable
    (1.0 + 2.0 ** -8, 0x3F80),  # midpoint between 1 and 1+2^-7 -> 1 (even)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),  # midpoint -> 1+2^-6 (even)
    (2.0 ** -133, 0x0001),      # smallest subnormal
    (2.0 ** -134, 0x0000),      # half the smallest subnormal -> 0 (even)
    (3 * 2.0 ** -135, 0x0001),  # 0.75 of the smallest subnormal -> it
    (3.3895313892515355e38, 0x7F7F),  # largest finite
    (3.4e38, 0x7F80),           # above max + half ulp -> inf
])
def test_bf16_hand_cases(v, bits):
    assert oracle.bf16_from_double(v) == bits
    assert _brute_bf16(v) == bits


def test_bf16_matches_torch_on_fp32_values():
    """Direct double->bf16 equals torch's fp32->bf16 when the input is an fp32."""
    rng = np.random.default_rng(1)
    raw = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    f = raw.view(np.float32)
    f = f[np.isfinite(f)]
    ties = (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    f = np.concatenate([f, ties, -ties, np.float32([1e-40, -1e-40, 3e38, -3e38])])
    ref = inputs.f32_to_bf16_bits(f)
    got = np.array([oracle.bf16_from_double(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_matches_brute_force_on_doubles():
    rng = np.random.default_rng(2)
    mags = rng.uniform(-140, 130, size=400)
    vals = np.sign(rng.standard_normal(400)) * 2.0 ** mags * rng.uniform(1, 2, size=400)
    for v in vals:
        assert oracle.bf16_from_double(float(v)) == _brute_bf16(float(v)), v


def test_bf16_roundtrip_all_patterns():
    for b in range(0, 0x10000, 7):
        if ((b >> 7) & 0xFF) == 0xFF:
            continue
        assert oracle.bf16_from_double(oracle.bf16_to_double(b)) == b


# --------------------------------------------------------- gate GEMM pins ---

def _as_fraction(bits: np.ndarray):
    return [Fraction(float(v)) for v in inputs.bf16_bits_to_f32(bits)]


def test_gate_logits_exact_on_tiny_inputs():
    rng = np.random.default_rng(3)
    M, H, E = 3, 24, 7
    x = inputs.f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32))
    w = inputs.f32_to_bf16_bits(rng.standard_normal((E, H)).astype(np.float32) * 0.02)
    bias = rng.standard_normal(E).astype(np.float32)
    z, ad = oracle.gate_logits(x, w, bias)
    for t in range(M):
        xf = _as_fraction(x[t])
        for e in range(E):
            wf = _as_fraction(w[e])
            exact = sum(a * b for a, b in zip(xf, wf)) + Fraction(float(bias[e]))
            assert abs(Fraction(z[t, e]) - exact) <= Fraction(2) ** -50 * abs(exact) + Fraction(2) ** -1000
            aexact = sum(abs(a * b) for a, b in zip(xf, wf)) + abs(Fraction(float(bias[e])))
            assert abs(Fraction(ad[t, e]) - aexact) <= Fraction(2) ** -50 * aexact


def test_gate_logits_match_numpy_matmul():
    rng = np.random.default_rng(4)
    M, H, E = 5, 512, 33
    x = inputs.f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32))
    w = inputs.f32_to_bf16_bits(rng.standard_normal((E, H)).astype(np.float32) * 0.02)
    z, _ = oracle.gate_logits(x, w)
    ref = inputs.bf16_bits_to_f32(x).astype(np.float64) @ inputs.bf16_bits_to_f32(w).astype(np.float64).T
    assert np.allclose(z, ref, rtol=1e-12, atol=1e-12)


def test_gate_logits_integer_inputs_exact():
    """Integer-valued bf16 entries in [-2,2]: every sum is an exact integer."""
    ri = inputs.make_route_inputs(2, 4096, 16, 4, 1, seed=5, dist="int")
    z, _ = oracle.gate_logits(ri.x, ri.w)
    ref = inputs.bf16_bits_to_f32(ri.x).astype(np.int64) @ inputs.bf16_bits_to_f32(ri.w).astype(np.int64).T
    assert np.array_equal(z, ref.astype(np.float64))


# ------------------------------------------------------- top-k / softmax ---

def _brute_select(zhat, k):
    order = sorted(range(len(zhat)), key=lambda e: (-zhat[e], e))[:k]
    return order


def test_select_matches_brute_force_with_ties():
    rng = np.random.default_rng(6)
    for trial in range(300):
        E = int(rng.integers(1, 24))
        k = int(rng.integers(1, E + 1))
        zhat = rng.integers(-3, 4, size=E).astype(np.float64) * 0.5
        ids, w = oracle.select(zhat, k)
        assert list(ids) == _brute_select(list(zhat), k)
        # weights: softmax over the selected, closed form in exact-ish double
        sel = zhat[ids]
        ref = np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum()
        assert np.allclose(w, ref.astype(np.float32), rtol=1e-7, atol=0)


def test_select_all_equal_lowest_ids_win():
    ids, w = oracle.select(np.zeros(512), 10)
    assert list(ids) == list(range(10))
    assert np.all(w == np.float32(0.1))


def test_select_signed_zero_ties_by_id():
    zhat = np.array([-1.0, -0.0, 0.0, -0.0, 0.0, -2.0])
    ids, w = oracle.select(zhat, 3)
    assert list(ids) == [1, 2, 3]
    assert np.all(w == np.float32(1 / 3))


def test_select_k1_weight_is_one():
    rng = np.random.default_rng(7)
    ids, w = oracle.select(rng.standard_normal(64), 1)
    assert w[0] == np.float32(1.0)


def test_select_k_equals_e_is_plain_softmax():
    rng = np.random.default_rng(8)
    zhat = oracle.bf16_round(rng.standard_normal(40) * 3)
    ids, w = oracle.select(zhat, 40)
    ref = scipy.special.softmax(zhat)[ids]
    assert np.allclose(w, ref, rtol=2e-7)
    assert list(ids) == list(np.lexsort((np.arange(40), -zhat)))


def test_select_two_experts_closed_form():
    a, b = 1.25, -0.5
    ids, w = oracle.select(np.array([b, a, -9.0]), 2)
    assert list(ids) == [1, 0]
    assert w[0] == np.float32(1.0 / (1.0 + math.exp(-(a - b))))
    assert w[1] == np.float32(1.0 / (1.0 + math.exp(a - b)))


def test_select_boundary_tie_takes_lower_id():
    zhat = np.array([5.0, 3.0, 4.0, 3.0, 3.0, 1.0])
    ids, _ = oracle.select(zhat, 3)
    assert list(ids) == [0, 2, 1]  # 3.0 appears at ids 1,3,4 -> id 1 wins


def test_shared_weight_closed_forms():
    assert oracle.shared_weight(0.0, 1.0) == np.float32(0.5)
    assert oracle.shared_weight(0.0, 2.5) == np.float32(1.25)
    for s in (-30.0, -3.0, -0.1, 0.7, 4.0, 20.0):
        assert oracle.shared_weight(s, 1.0) == np.float32(scipy.special.expit(s))


# -------------------------------------------------------------- full route ---

def test_route_invariants_and_shared_slot():
    ri = inputs.make_route_inputs(6, 256, 64, 5, 1, seed=9, shared_scale=1.5)
    r = oracle.route(ri.x, ri.w, ri.ws, None, ri.topk, ri.shared_scale)
    assert r.ids.shape == (6, 6)
    for t in range(6):
        routed = r.ids[t, :5]
        assert len(set(routed)) == 5 and routed.max() < 64 and routed.min() >= 0
        assert abs(float(r.w[t, :5].astype(np.float64).sum()) - 1.0) < 1e-6
        assert r.ids[t, 5] == 64
        s_ref = float(inputs.bf16_bits_to_f32(ri.x[t]).astype(np.float64)
                      @ inputs.bf16_bits_to_f32(ri.ws[0]).astype(np.float64))
        assert r.w[t, 5] == np.float32(1.5 * scipy.special.expit(s_ref))
        # selected values are the k largest rounded logits
        zh = r.zhat[t]
        kth = zh[routed[-1]]
        assert np.all(zh[routed] >= kth)
        others = np.setdiff1d(np.arange(64), routed)
        assert np.all(zh[others] <= kth)


def test_route_zero_shared_gate_gives_half_scale():
    ri = inputs.make_route_inputs(3, 128, 16, 2, 1, seed=10, shared_scale=3.0)
    ri.ws[:] = 0
    r = oracle.route(ri.x, ri.w, ri.ws, None, 2, 3.0)
    assert np.all(r.w[:, 2] == np.float32(1.5))


def test_route_rounds_logits_before_topk():
    """A one-hot gate builds logits 257 and 256.5: 257 rounds to 256 in bf16,
    so the two experts tie and the lower id wins even though 257 > 256.5."""
    H, E = 8, 3
    x = inputs.f32_to_bf16_bits(np.array([[1, 0, 0, 0, 0, 0, 0, 0]], np.float32))
    w = np.zeros((E, H), np.uint16)
    w[0, 0] = inputs.f32_to_bf16_bits(np.float32([256.0]))[0]
    w[1, 0] = inputs.f32_to_bf16_bits(np.float32([256.0]))[0]
    bias = np.array([0.5, 1.0, 0.0], np.float32)  # z = 256.5 (-> 256), 257 (-> 256)
    r = oracle.route(x, w, None, bias, 1)
    assert r.zhat[0, 0] == 256.0 and r.zhat[0, 1] == 256.0
    assert r.ids[0, 0] == 0
    bias2 = np.array([0.5, 3.0, 0.0], np.float32)  # 259 -> 260 beats 256
    r2 = oracle.route(x, w, None, bias2, 1)
    assert r2.zhat[0, 1] == 260.0 and r2.ids[0, 0] == 1


def test_route_bias_added_before_rounding():
    rng = np.random.default_rng(11)
    ri = inputs.make_route_inputs(4, 64, 32, 4, 0, seed=12, zipf_s=1.1)
    r = oracle.route(ri.x, ri.w, None, ri.bias, 4)
    z, _ = oracle.gate_logits(ri.x, ri.w)
    assert np.allclose(r.z, z + ri.bias.astype(np.float64)[None, :], rtol=0, atol=1e-12)
    assert np.array_equal(r.zhat, oracle.bf16_round(r.z))


# ------------------------------------------------------------------- align ---

def _textbook_align(ids, E_al, A):
    flat = np.asarray(ids, np.int64).ravel()
    numel = flat.size
    order = np.argsort(flat, kind="stable")
    cnt = np.bincount(flat, minlength=E_al)
    padded = (cnt + A - 1) // A * A
    off = np.concatenate([[0], np.cumsum(padded)])
    out = np.full(off[-1], numel, np.int64)
    start = np.concatenate([[0], np.cumsum(cnt)])
    eid = []
    for e in range(E_al):
        out[off[e]: off[e] + cnt[e]] = order[start[e]: start[e + 1]]
        eid += [e] * (padded[e] // A)
    return out, np.array(eid, np.int64), int(off[-1])


@pytest.mark.parametrize("T,W,E_al,A,skew", [
    (1, 1, 1, 1, None), (4, 11, 513, 64, None), (37, 8, 128, 64, 1.1),
    (200, 8, 128, 128, None), (64, 3, 7, 5, 2.0), (300, 11, 513, 128, 1.1),
])
def test_align_matches_stable_argsort(T, W, E_al, A, skew):
    ids = inputs.random_ids(T, W, E_al, seed=T * 7 + A, skew=skew)
    r = oracle.align(ids, E_al, A)
    ref_sorted, ref_eid, ref_npp = _textbook_align(ids, E_al, A)
    assert r.npp == ref_npp
    assert np.array_equal(r.sorted_ids, ref_sorted)
    assert np.array_equal(r.expert_ids, ref_eid)


def test_align_invariants():
    ids = inputs.random_ids(500, 11, 513, seed=13, skew=1.1)
    A = 64
    r = oracle.align(ids, 513, A)
    numel = ids.size
    real = r.sorted_ids[r.sorted_ids < numel]
    assert np.array_equal(np.sort(real), np.arange(numel))          # each slot once
    assert r.npp % A == 0
    cnt = np.bincount(ids.ravel(), minlength=513)
    assert r.npp == int(((cnt + A - 1) // A * A).sum())            # ceil-sum formula
    assert np.all(np.diff(r.expert_ids) >= 0)                       # non-decreasing
    blocks = r.sorted_ids.reshape(-1, A)
    for b, e in enumerate(r.expert_ids):                            # block purity
        rows = blocks[b][blocks[b] < numel]
        assert np.all(ids.ravel()[rows] == e)
    assert r.npp <= oracle.align_capacity(numel, 513, A)


def test_align_single_expert_edge_cases():
    A = 64
    r = oracle.align(np.full(A, 5, np.int32), 8, A)
    assert r.npp == A and list(r.expert_ids) == [5]
    assert np.array_equal(r.sorted_ids, np.arange(A))
    r = oracle.align(np.full(A + 1, 5, np.int32), 8, A)
    assert r.npp == 2 * A and list(r.expert_ids) == [5, 5]
    assert np.array_equal(r.sorted_ids[: A + 1], np.arange(A + 1))
    assert np.all(r.sorted_ids[A + 1:] == A + 1)                    # sentinel = numel
    r = oracle.align(np.zeros(0, np.int32), 8, A)
    assert r.npp == 0


def test_align_capacity_printed_values():
    for toks, k, E, A, slots in _golden("align_capacity.txt"):
        assert oracle.align_capacity(int(toks) * int(k), int(E), int(A)) == int(slots)


def test_block_size_tier_printed_values():
    for toks, k, E, A in _golden("block_size_tier.txt"):
        assert oracle.select_block_size(int(toks), int(k), int(E)) == int(A)


def test_block_size_tier_tracks_e_and_k():
    # the threshold is one 128-row block of routed rows per expert
    assert oracle.select_block_size(1024, 8, 64) == 128      # exactly 128 rows per expert
    assert oracle.select_block_size(1023, 8, 64) == 64
    assert oracle.select_block_size(2047, 8, 128) == 64
    assert oracle.select_block_size(4096, 10, 512) == 64     # 80 rows per expert
    assert oracle.select_block_size(16384, 10, 512) == 128   # 320 rows per expert


def _routing_with_touched(tokens, k, E, touched, seed):
    """Rows of k distinct experts drawn from exactly `touched` experts."""
    rng = np.random.default_rng(seed)
    pool = rng.permutation(E)[:touched]
    ids = np.empty((tokens, k), np.int32)
    need = list(pool)
    for t in range(tokens):
        row = need[:k]
        need = need[k:]
        rest = [e for e in rng.permutation(pool) if e not in row][: k - len(row)]
        ids[t] = np.array(row + rest, np.int32)
    assert len(np.unique(ids)) == touched
    return ids


def test_npp_table_single_block_rows():
    """Where every touched expert fits in one block, npp = touched * A; the
    page's rows for 6 tokens (both A) and 128 tokens (A=128) are of that kind."""
    rows = {int(r[0]): r for r in _golden("npp_table.txt")}
    toks, touched, npp64, npp128 = (int(v) for v in rows[6][:4])
    ids = _routing_with_touched(toks, 8, 128, touched, seed=14)
    assert oracle.align(ids, 128, 64).npp == npp64
    assert oracle.align(ids, 128, 128).npp == npp128
    toks, touched, _, npp128 = (int(v) for v in rows[128][:4])
    ids = _routing_with_touched(toks, 8, 128, touched, seed=15)
    assert oracle.align(ids, 128, 128).npp == npp128


def test_npp_table_ratio_is_npp_over_routed_rows():
    for toks, touched, npp64, npp128, ratio in _golden("npp_table.txt"):
        assert round(int(npp128) / (int(toks) * 8), 1) == float(ratio)
        # averages of per-layer multiples of A, never below one block per touched expert
        assert int(npp64) * 4 % 64 == 0 and int(npp128) * 4 % 128 == 0
        assert int(npp128) >= int(touched) * 128 and int(npp64) >= int(touched) * 64


# ------------------------------------------------------- routing variants ---

def test_select_without_renormalisation_is_the_full_softmax_at_the_top_k():
    """renormalize = 0: the weights are scipy's softmax over all E logits,
    read at the selected ids (same ids as with renormalisation)."""
    rng = np.random.default_rng(41)
    for E, k in ((64, 8), (513, 10), (7, 3)):
        z = oracle.bf16_round(rng.normal(0, 2, E))
        ids, w = oracle.select(z, k, renormalize=False)
        ids1, w1 = oracle.select(z, k)
        assert np.array_equal(ids, ids1)
        ref = scipy.special.softmax(z)[ids]
        assert np.allclose(w, ref.astype(np.float32), rtol=1.2e-7, atol=0)
        assert float(w.astype(np.float64).sum()) < 1.0
        # renormalising the unrenormalised weights gives the renormalised ones
        assert np.allclose(w / w.astype(np.float64).sum(), w1, rtol=1e-6)


def test_select_without_renormalisation_k_equals_e():
    z = oracle.bf16_round(np.random.default_rng(42).normal(0, 1, 16))
    ids0, w0 = oracle.select(z, 16, renormalize=False)
    ids1, w1 = oracle.select(z, 16)
    assert np.array_equal(ids0, ids1) and np.array_equal(w0, w1)


def test_route_without_renormalisation():
    ri = inputs.make_route_inputs(5, 256, 64, 6, 1, seed=43)
    r0 = oracle.route(ri.x, ri.w, ri.ws, None, 6, renormalize=False)
    r1 = oracle.route(ri.x, ri.w, ri.ws, None, 6)
    assert np.array_equal(r0.ids, r1.ids)
    for t in range(5):
        ref = scipy.special.softmax(r0.zhat[t])[r0.ids[t, :6]]
        assert np.allclose(r0.w[t, :6], ref.astype(np.float32), rtol=1.2e-7, atol=0)
    assert np.array_equal(r0.w[:, 6], r1.w[:, 6])  # the shared slot is unaffected


def test_route_shared_logit_rounded_to_bf16():
    """shared_bf16: a shared logit of exactly 1 + 2^-9 rounds to 1.0 first, so
    the weight is expit(1.0) rather than expit(1 + 2^-9); without the flag it
    is the latter. Routed outputs do not change."""
    H, E = 8, 4
    x = inputs.f32_to_bf16_bits(np.array([[1, 1, 0, 0, 0, 0, 0, 0]], np.float32))
    ws = inputs.f32_to_bf16_bits(np.array([[1, 2.0 ** -9, 0, 0, 0, 0, 0, 0]], np.float32))
    w = inputs.f32_to_bf16_bits(np.eye(E, H, dtype=np.float32))
    r1 = oracle.route(x, w, ws, None, 2, 2.0, shared_bf16=True)
    r0 = oracle.route(x, w, ws, None, 2, 2.0)
    assert r1.s[0] == 1.0 + 2.0 ** -9
    assert r1.w[0, 2] == np.float32(2.0 * scipy.special.expit(1.0))
    assert r0.w[0, 2] == np.float32(2.0 * scipy.special.expit(1.0 + 2.0 ** -9))
    assert r0.w[0, 2] != r1.w[0, 2]
    assert np.array_equal(r0.ids, r1.ids) and np.array_equal(r0.w[:, :2], r1.w[:, :2])


def test_align_eplb_identity_map_is_plain_align():
    ids = inputs.random_ids(300, 9, 65, seed=44, skew=1.1)
    mp = np.arange(65, dtype=np.int32)[:, None]
    got = oracle.align_eplb(ids, 65, mp, np.ones(65, np.int32), 65, 16)
    ref = oracle.align(ids, 65, 16)
    assert got.npp == ref.npp
    assert np.array_equal(got.sorted_ids, ref.sorted_ids) and np.array_equal(got.expert_ids, ref.expert_ids)


def test_align_eplb_permutation_is_a_relabelling():
    """One replica per expert, physical ids a permutation over more physical
    slots: the same as aligning the relabelled ids (numpy take), with the
    unused physical experts empty."""
    rng = np.random.default_rng(45)
    ids = inputs.random_ids(200, 5, 40, seed=46)
    perm = rng.permutation(48)[:40].astype(np.int32)
    got = oracle.align_eplb(ids, 40, perm[:, None], np.ones(40, np.int32), 48, 8)
    ref = _textbook_align(np.take(perm, ids), 48, 8)
    assert got.npp == len(ref[0])
    assert np.array_equal(got.sorted_ids, ref[0]) and np.array_equal(got.expert_ids, ref[1])


def test_align_eplb_replicas_hand_case():
    """Hand-worked: 4 tokens x 2 slots, expert 0 held by physical 5 and 2
    (two replicas), expert 1 by physical 3, expert 2 by physical 0; A = 2.
    Token t's slot of expert 0 goes to replica t mod 2 (tokens 2 and 3 hold
    expert 0 in different slot positions, so the token, not the slot, picks):
      ids   [[0,1],[2,0],[1,0],[0,2]]  (flat 0..7)
      phys  [[5,3],[0,2],[3,5],[2,0]]
    physical 0: flat 2, 7; physical 2: flat 3, 6; physical 3: flat 1, 4;
    physical 5: flat 0, 5."""
    ids = np.array([[0, 1], [2, 0], [1, 0], [0, 2]], np.int32)
    mp = np.array([[5, 2], [3, -1], [0, -1]], np.int32)
    cnt = np.array([2, 1, 1], np.int32)
    got = oracle.align_eplb(ids, 3, mp, cnt, 6, 2)
    assert got.npp == 8
    assert got.sorted_ids.tolist() == [2, 7, 3, 6, 1, 4, 0, 5]
    assert got.expert_ids.tolist() == [0, 2, 3, 5]
    # a replica count above the table width is refused
    with pytest.raises(ValueError):
        oracle.align_eplb(ids, 3, mp, np.array([3, 1, 1], np.int32), 6, 2)


# ------------------------------------------------ hidden states to e4m3 ---

def _e4m3_table():
    """All finite e4m3 values except -0, as (Fraction, code), sorted."""
    out = []
    for c in range(256):
        if (c & 0x7F) == 0x7F or c == 0x80:
            continue
        ef, fr = (c >> 3) & 0xF, c & 7
        mag = Fraction(fr, 8) * Fraction(1, 64) if ef == 0 else (1 + Fraction(fr, 8)) * Fraction(2) ** (ef - 7)
        out.append((-mag if c & 0x80 else mag, c))
    return sorted(out)


def test_e4m3_exhaustive_brute_force():
    """Every code, every midpoint between neighbours (ties to the even code)
    and points just beside the midpoints, against exact rationals."""
    table = _e4m3_table()
    assert len(table) == 253 and table[-1][0] == 448 and table[0][0] == -448
    for v, c in table:
        assert oracle.e4m3_from_double(float(v)) == c
        assert oracle.e4m3_to_double(c) == float(v)
    for (a, ca), (b, cb) in zip(table, table[1:]):
        mid = (a + b) / 2
        even = ca if (ca & 1) == 0 else cb
        if a == 0 or b == 0:  # around zero the sign of the rounded zero follows v
            continue
        assert oracle.e4m3_from_double(float(mid)) == even, (a, b)
        eps = (b - a) / 1024
        assert oracle.e4m3_from_double(float(mid - eps)) == ca
        assert oracle.e4m3_from_double(float(mid + eps)) == cb


def test_e4m3_saturates_and_matches_torch():
    for v, c in ((448.0, 0x7E), (449.0, 0x7E), (479.9, 0x7E), (1e9, 0x7E), (-500.0, 0xFE),
                 (2.0 ** -10, 0x00), (3 * 2.0 ** -11, 0x01)):
        assert oracle.e4m3_from_double(v) == c, v
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(71)
    v = np.concatenate([rng.uniform(-447, 447, 4000), rng.normal(0, 1, 4000),
                        rng.normal(0, 0.01, 2000)]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_double(float(x)) for x in v], np.uint8)
    assert np.array_equal(got, ref)


def test_quant_fp8_closed_forms():
    """A block whose largest magnitude is a: scale = fl(a / 448), that
    element's code is +-448, a zero block gives scale 0 and zero codes,
    every code decodes within half an e4m3 step of x * 448 / a."""
    H = 256
    xf = np.zeros((2, H), np.float32)
    xf[0, :128] = np.linspace(-3.0, 2.5, 128)
    xf[1, 128:] = np.random.default_rng(72).normal(0, 1, 128)
    x = inputs.f32_to_bf16_bits(xf)
    xv = inputs.bf16_bits_to_f32(x).astype(np.float64)
    q, sc = oracle.quant_fp8(x)
    assert sc[0, 1] == 0.0 and np.all(q[0, 128:] == 0) and sc[1, 0] == 0.0 and np.all(q[1, :128] == 0)
    for t, b in ((0, 0), (1, 1)):
        blk = xv[t, 128 * b:128 * b + 128]
        a = np.abs(blk).max()
        assert sc[t, b] == np.float32(a / 448.0)
        i = int(np.argmax(np.abs(blk)))
        assert oracle.e4m3_to_double(q[t, 128 * b + i]) == math.copysign(448.0, blk[i])
        dec = np.array([oracle.e4m3_to_double(c) for c in q[t, 128 * b:128 * b + 128]])
        scaled = blk * (448.0 / a)
        step = np.where(np.abs(scaled) < 2.0 ** -6, 2.0 ** -9,
                        2.0 ** (np.floor(np.log2(np.maximum(np.abs(scaled), 1e-30))) - 3))
        assert np.all(np.abs(dec - scaled) <= step / 2 * (1 + 1e-6) + 1e-9)


# ---------------------------------------------------- consumer expert GEMM ---

def test_expert_gemm_matches_numpy_per_expert():
    """Each slot's row equals x[token] @ W[expert].T (numpy fp64 matmul)."""
    rng = np.random.default_rng(81)
    T, width, E, N, H = 7, 3, 5, 16, 64
    x = inputs.f32_to_bf16_bits(rng.normal(0, 1, (T, H)).astype(np.float32))
    w = inputs.f32_to_bf16_bits(rng.normal(0, 0.05, (E, N, H)).astype(np.float32))
    ids = inputs.random_ids(T, width, E, seed=82)
    out, ad = oracle.expert_gemm(x, ids, w)
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    wf = inputs.bf16_bits_to_f32(w).astype(np.float64)
    ref = np.einsum("th,tsnh->tsn", xf, wf[ids]).reshape(T * width, N)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    aref = np.einsum("th,tsnh->tsn", np.abs(xf), np.abs(wf[ids])).reshape(T * width, N)
    assert np.allclose(ad, aref, rtol=1e-12, atol=0)


def test_expert_gemm_integer_inputs_exact():
    """Integer entries: every product and sum is exact in double."""
    rng = np.random.default_rng(83)
    T, width, E, N, H = 5, 2, 3, 8, 128
    x = inputs.f32_to_bf16_bits(rng.integers(-3, 4, (T, H)).astype(np.float32))
    w = inputs.f32_to_bf16_bits(rng.integers(-3, 4, (E, N, H)).astype(np.float32))
    ids = np.array([[0, 2], [1, 0], [2, 1], [0, 1], [2, 0]], np.int32)
    out, _ = oracle.expert_gemm(x, ids, w)
    xi = inputs.bf16_bits_to_f32(x).astype(np.int64)
    wi = inputs.bf16_bits_to_f32(w).astype(np.int64)
    for t in range(T):
        for s in range(width):
            assert np.array_equal(out[t * width + s], (wi[ids[t, s]] @ xi[t]).astype(np.float64))
