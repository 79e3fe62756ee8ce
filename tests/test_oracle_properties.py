"""Property pins for the CPU oracle (hypothesis draws the cases; skipped where
hypothesis is not installed). Each property restates a definition from the
pages in its plainest form and checks the oracle against it:

- moe_align_block_size ("[ROCm][Kernel] W4A16 MoE prefill: M-aware moe_align
  block size", Purpose): every expert's ids in ascending flat order, padded
  to a multiple of A with the sentinel numel, experts in ascending order, one
  expert id per block;
- top-k ("[AMD] One-launch small-M MoE router for Qwen3.5 on gfx950",
  Modifications): the k largest rounded logits, ties to the lowest id, slots
  in (value desc, id asc) order, with softmax weights renormalised over them.
CPU only.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
given, settings = hyp.given, hyp.settings


def _align_by_definition(flat: np.ndarray, E_al: int, A: int):
    """Padded, expert-grouped list built directly from the definition."""
    out, owners = [], []
    n = flat.shape[0]
    for e in range(E_al):
        mine = [i for i in range(n) if flat[i] == e]  # ascending flat order
        if not mine:
            continue
        blocks = -(-len(mine) // A)
        out += mine + [n] * (blocks * A - len(mine))
        owners += [e] * blocks
    return np.array(out, dtype=np.int32), np.array(owners, dtype=np.int32)


@settings(max_examples=150, deadline=None)
@given(T=st.integers(0, 40), W=st.integers(1, 6), E_al=st.integers(1, 20), A=st.integers(1, 9),
       seed=st.integers(0, 2**31 - 1))
def test_align_matches_its_definition(T, W, E_al, A, seed):
    rng = np.random.default_rng(seed)
    # a few hot experts make multi-block experts and empty experts likely
    hot = rng.integers(0, E_al, size=min(3, E_al))
    ids = np.where(rng.random((T, W)) < 0.5, rng.choice(hot, size=(T, W)),
                   rng.integers(0, E_al, size=(T, W))).astype(np.int32)
    res = oracle.align(ids, E_al, A)
    want_sorted, want_owner = _align_by_definition(ids.ravel(), E_al, A)
    assert res.npp == want_sorted.shape[0]
    assert res.npp % A == 0
    assert res.npp <= oracle.align_capacity(T * W, E_al, A)
    assert np.array_equal(res.sorted_ids, want_sorted)
    assert np.array_equal(res.expert_ids, want_owner)


@settings(max_examples=150, deadline=None)
@given(E=st.integers(1, 24), data=st.data())
def test_select_matches_its_definition(E, data):
    k = data.draw(st.integers(1, E))
    # few distinct values (many ties), signed zeros included
    pool = [-3.0, -1.5, -0.0, 0.0, 0.5, 2.0, 2.0, 7.25]
    z = np.array(data.draw(st.lists(st.sampled_from(pool), min_size=E, max_size=E)), dtype=np.float64)
    ids, w = oracle.select(z, k)
    # the k largest values, ties (and -0 == +0) to the lowest id, in that order
    want = sorted(range(E), key=lambda e: (-z[e], e))[:k]
    assert list(ids) == want
    m = max(z[e] for e in want)
    ex = [math.exp(z[e] - m) for e in want]
    den = math.fsum(ex)
    for j, e in enumerate(want):
        ref = np.float32(ex[j] / den)  # fp64 softmax rounded once to fp32; sums may
        assert abs(w[j] - ref) <= np.spacing(ref)  # associate differently: 1 ulp
