"""The GPU comparison rules (tests/_parity.py) are not vacuous: results built
from the oracle pass them, and the same results with one planted error are
rejected. CPU only (no kernel runs here: the 'GPU' outputs are the oracle's
own, then perturbed)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from moe_router_top_gb300 import inputs

from _parity import check_align, check_route, check_route_properties


def _oracle_outputs(ri):
    ref = oracle.route(ri.x, ri.w, ri.ws, ri.bias, ri.topk, ri.shared_scale)
    bits = np.array([[oracle.bf16_from_double(v) for v in row] for row in ref.zhat], dtype=np.uint16)
    return ref.ids.copy(), ref.w.copy(), bits


@pytest.fixture(scope="module")
def case():
    ri = inputs.make_route_inputs(6, 256, 64, 8, 1, seed=910, shared_scale=0.75)
    return ri, _oracle_outputs(ri)


def test_oracle_outputs_pass(case):
    ri, (ids, w, bits) = case
    for lg in (bits, None):  # with and without the GPU's logits
        rep = check_route(ri, ids, w, lg)
        assert rep.exact_rows == rep.rows and rep.rounding_rows == 0 and rep.logit_mismatch == 0
    check_route_properties(ri, ids, w)


def _flip_case(ri, monkeypatch, rel):
    """Widen the admissible band (accumulation_bound -> rel) so that logits of
    the oracle's top-k have two admissible roundings; returns a row, a
    selected expert whose logit can round the other way, and that value."""
    import _parity
    monkeypatch.setattr(_parity, "accumulation_bound", lambda _ri: rel)
    ref = oracle.route(ri.x, ri.w, ri.ws, ri.bias, ri.topk, ri.shared_scale)
    lo = oracle.bf16_round(ref.z - rel * ref.absdot)
    hi = oracle.bf16_round(ref.z + rel * ref.absdot)
    for t in range(ri.M):
        for e in ref.ids[t, :ri.topk]:
            if lo[t, e] != hi[t, e]:
                alt = hi[t, e] if ref.zhat[t, e] == lo[t, e] else lo[t, e]
                return ref, t, int(e), alt
    raise AssertionError("no selected logit near a rounding boundary")


def test_admissible_rounding_flip_is_accepted_and_counted(case, monkeypatch):
    """A result that the oracle's selection produces on an admissible
    rounding of one selected logit is accepted as a rounding row, with and
    without the GPU's logits; an unexplained one is not."""
    ri, (ids0, w0, bits0) = case
    ref, t, e, alt = _flip_case(ri, monkeypatch, 2.0 ** -13)
    z = ref.zhat[t].copy()
    z[e] = alt
    sid, sw = oracle.select(z, ri.topk)
    ids, w, bits = ids0.copy(), w0.copy(), bits0.copy()
    ids[t, :ri.topk], w[t, :ri.topk] = sid, sw
    bits[t, e] = oracle.bf16_from_double(alt)
    for lg in (bits, None):
        rep = check_route(ri, ids, w, lg)
        assert rep.rounding_rows == 1 and rep.exact_rows == ri.M - 1
    w[t, 0] *= 1 + 1e-5  # no admissible rounding gives this weight
    with pytest.raises(AssertionError):
        check_route(ri, ids, w, None)


def test_expert_change_off_the_boundary_is_rejected(case):
    """A different expert SET is accepted only on boundary rows (the oracle's
    k-th and (k+1)-th logits within 1 ulp), whatever else would explain it."""
    ri, (ids0, w0, bits0) = case
    ref = oracle.route(ri.x, ri.w, ri.ws, ri.bias, ri.topk, ri.shared_scale)
    k = ri.topk
    zs = -np.sort(-ref.zhat, axis=1)
    t = int(np.argmax(zs[:, k - 1] - zs[:, k]))  # the row farthest from a boundary tie
    z = ref.zhat[t].copy()
    out = int(np.argsort(-z, kind="stable")[k])  # the (k+1)-th expert enters the top-k
    z[out] = zs[t, 0] + 1.0
    sid, sw = oracle.select(z, k)
    ids, w = ids0.copy(), w0.copy()
    ids[t, :k], w[t, :k] = sid, sw
    with pytest.raises(AssertionError, match="off the k-th boundary"):
        check_route(ri, ids, w, None)


@pytest.mark.parametrize("mistake", [
    "swap two routed slots",       # slot order (value desc, id asc)
    "replace a routed expert",     # a wrong choice
    "weight off by 1e-5",          # beyond 2e-6 relative
    "shared slot id",              # slot k must be E
    "shared weight off by 1e-5",
    "logit two bf16 steps away",   # outside the accumulation bound
])
def test_route_rules_reject(case, mistake):
    ri, (ids, w, bits) = case
    ids, w, bits = ids.copy(), w.copy(), bits.copy()
    k = ri.topk
    if mistake == "swap two routed slots":
        ids[2, [0, 1]] = ids[2, [1, 0]]
    elif mistake == "replace a routed expert":
        unused = sorted(set(range(ri.E)) - set(ids[3, :k].tolist()))
        ids[3, k - 1] = unused[-1]
    elif mistake == "weight off by 1e-5":
        w[1, 0] *= 1 + 1e-5
    elif mistake == "shared slot id":
        ids[0, k] = ri.E - 1
    elif mistake == "shared weight off by 1e-5":
        w[4, k] *= 1 + 1e-5
    elif mistake == "logit two bf16 steps away":
        e = int(ids[5, 0])
        bits[5, e] = bits[5, e] + 2 if bits[5, e] < 0x8000 else bits[5, e] - 2
    with pytest.raises(AssertionError):
        check_route(ri, ids, w, bits)
    if mistake != "logit two bf16 steps away":  # the same mistake without the GPU's logits
        with pytest.raises(AssertionError):
            check_route(ri, ids, w, None)


@pytest.fixture(scope="module")
def align_case():
    ids = inputs.random_ids(40, 5, 17, seed=911, skew=1.1)
    ref = oracle.align(ids, 17, 4)
    cap = oracle.align_capacity(ids.size, 17, 4)
    srt = np.full(cap, -1, np.int32)
    srt[: ref.npp] = ref.sorted_ids
    eids = np.full((cap + 3) // 4, -1, np.int32)
    eids[: ref.npp // 4] = ref.expert_ids
    return ids, ref, srt, eids


def test_oracle_align_passes(align_case):
    ids, ref, srt, eids = align_case
    check_align(ids, 17, 4, srt, eids, np.array([ref.npp], np.int32))


@pytest.mark.parametrize("mistake", ["npp one block short", "two ids swapped", "sentinel wrong",
                                     "block owner wrong"])
def test_align_rules_reject(align_case, mistake):
    ids, ref, srt, eids = align_case
    srt, eids, npp = srt.copy(), eids.copy(), ref.npp
    if mistake == "npp one block short":
        npp -= 4
    elif mistake == "two ids swapped":
        real = np.nonzero(ref.sorted_ids < ids.size)[0]  # positions holding ids, not padding
        i, j = int(real[0]), int(real[1])                 # distinct flat indices
        srt[[i, j]] = srt[[j, i]]
    elif mistake == "sentinel wrong":
        p = int(np.argmax(ref.sorted_ids == ids.size))
        srt[p] = 0
    elif mistake == "block owner wrong":
        eids[0] = (eids[0] + 1) % 17
    with pytest.raises(AssertionError):
        check_align(ids, 17, 4, srt, eids, np.array([npp], np.int32))


def _fp32_chain_route(ri, renormalize=True):
    """A stand-in for an fp32-accumulating kernel: the dot of every 16-wide
    K block exactly, the blocks added one by one in fp32 (H/16 additions, the
    tcgen05 path's chain), the bias added in fp32, then the oracle's bf16
    rounding and selection."""
    x = inputs.bf16_bits_to_f32(ri.x).astype(np.float64)
    w = inputs.bf16_bits_to_f32(ri.w).astype(np.float64)
    acc = np.zeros((ri.M, ri.E), np.float32)
    for c in range(0, ri.H, 16):
        acc = (acc + (x[:, c:c + 16] @ w[:, c:c + 16].T).astype(np.float32)).astype(np.float32)
    if ri.bias is not None:
        acc = (acc + ri.bias).astype(np.float32)
    return oracle.select_rows(oracle.bf16_round(acc.astype(np.float64)), ri.topk, renormalize)


@pytest.mark.parametrize("renormalize", [True, False])
@pytest.mark.parametrize("M", [1024, 2048])
def test_fp32_accumulation_stand_in_passes(M, renormalize):
    """Results of a real fp32 accumulation order differ from the fp64
    oracle's on a few rows (a logit rounds the other way); the rule must
    accept and count them, and reject none."""
    ri = inputs.zipf_sweep(M)
    ri.renormalize = renormalize
    ids, w = _fp32_chain_route(ri, renormalize)
    rep = check_route(ri, ids, w, None)
    assert rep.rounding_rows >= 1 and rep.set_differs_rows == 0
