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
    rep = check_route(ri, ids, w, bits)
    check_route_properties(ri, ids, w)
    assert rep.rows_ids_differ == 0 and rep.logit_mismatch == 0


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
