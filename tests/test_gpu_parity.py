"""GPU parity: the CUDA path (through the C ABI) against the oracle on the five
workloads, edge cases, graph replay and workspace reuse. Needs a GB300.

The workloads are checked twice: as the benchmark calls route_align (no
logits output, the benchmark's block sizes and a reused workspace), and with
the optional logits output, whose every value is then checked against the
accumulation bound. Each comparison's counts (exact, rounding-flip, boundary
and near-midpoint rows) are appended to $SMR_PARITY_LOG when it is set.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from moe_router_top_gb300 import inputs

from _parity import check_align, check_route, check_route_properties, record

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def smr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import moe_router_top_gb300 as m
    return m


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _dev(ri):
    x = _bf16(ri.x)
    w = _bf16(ri.w)
    ws = _bf16(ri.ws) if ri.ws is not None else None
    b = torch.from_numpy(ri.bias).cuda() if ri.bias is not None else None
    return x, w, ws, b


def _route_align(smr, ri, A, with_logits=True, workspace=None):
    x, w, ws, b = _dev(ri)
    logits = torch.empty((ri.M, ri.E), dtype=torch.int16, device="cuda") if with_logits else None
    out = smr.route_align(x, w, ws, b, topk=ri.topk, block_size=A, shared_scale=ri.shared_scale,
                          logits_out=logits, workspace=workspace)
    torch.cuda.synchronize()
    ids, wts, srt, eids, npp = (t.cpu().numpy() for t in out)
    lg = logits.cpu().numpy().view(np.uint16) if with_logits else None
    return ids, wts, srt, eids, npp, lg


def _full_check(smr, ri, A, exact=False, with_logits=True, name=None):
    ids, wts, srt, eids, npp, lg = _route_align(smr, ri, A, with_logits=with_logits)
    rep = check_route(ri, ids, wts, lg, exact_logits=exact)
    check_route_properties(ri, ids, wts)
    Aeff = A if A > 0 else oracle.select_block_size(ri.M, ri.topk, ri.E)
    al = check_align(ids, ri.num_experts_align, Aeff, srt, eids, npp)
    if name:
        record(name, rep, logits_out=with_logits, npp=al.npp, block_size=Aeff)
    return rep, al, ids


# ------------------------------------------------------------- workloads --

@pytest.mark.parametrize("with_logits", [False, True], ids=["bench_call", "logits_out"])
@pytest.mark.parametrize("M", [4, 8])
def test_small_verify(smr, M, with_logits):
    """M=4 (and 8), as bench.py times it: one single-launch route_align with
    A=64 (and the same with the logits output)."""
    ri = inputs.small_verify(M)
    rep, al, _ = _full_check(smr, ri, 64, with_logits=with_logits,
                             name=f"small_verify_M{M}" + ("_logits" if with_logits else ""))
    assert smr.last_launch_count() == 1
    print(f"small_verify M={M}: {rep} npp={al.npp}")


@pytest.mark.parametrize("with_logits", [False, True], ids=["bench_call", "logits_out"])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_tie_stress_bit_exact(smr, M, with_logits):
    """Integer inputs: fp32 accumulation is exact, so every logit, id and
    align output must match the oracle bit for bit."""
    ri = inputs.tie_stress(M)
    rep, al, ids = _full_check(smr, ri, 64, exact=True, with_logits=with_logits,
                               name=f"tie_stress_M{M}" + ("_logits" if with_logits else ""))
    assert rep.exact_rows == rep.rows


@pytest.mark.parametrize("with_logits", [False, True], ids=["bench_call", "logits_out"])
def test_short_prefill_blocks(smr, with_logits):
    ri = inputs.short_prefill()
    res = {}
    for A in (64, 128, 0):
        rep, al, ids = _full_check(smr, ri, A, with_logits=with_logits,
                                   name=f"short_prefill_A{A}" + ("_logits" if with_logits else ""))
        res[A] = al.npp
    assert oracle.select_block_size(128, 8, 128) == 64 and res[0] == res[64]
    print(f"short_prefill npp: A=64 {res[64]}, A=128 {res[128]}, ratio@128 {res[128] / 1024:.2f}")


@pytest.mark.parametrize("with_logits", [False, True], ids=["bench_call", "logits_out"])
@pytest.mark.parametrize("M", list(inputs.ZIPF_TOKENS))
def test_zipf_sweep(smr, M, with_logits):
    ri = inputs.zipf_sweep(M)
    rep, al, ids = _full_check(smr, ri, 0, with_logits=with_logits,
                               name=f"zipf_M{M}" + ("_logits" if with_logits else ""))
    A = oracle.select_block_size(M, 8, 128)
    cnt = np.bincount(ids.ravel(), minlength=128)
    assert al.npp == int(((cnt + A - 1) // A * A).sum())
    print(f"zipf M={M}: A={A} npp={al.npp} touched={(cnt > 0).sum()} {rep}")


def test_large_batch_bench_call_all_rows(smr):
    """M=16384 exactly as bench.py calls it (route_align, A=128, no logits
    output, a reused workspace, second call on it): EVERY row against the
    oracle (row-parallel on the host cores), invariants on all rows, align
    bit-exact on all ids."""
    ri = inputs.large_batch()
    wsp = smr.Workspace()
    _route_align(smr, ri, 128, with_logits=False, workspace=wsp)
    ids, wts, srt, eids, npp, _ = _route_align(smr, ri, 128, with_logits=False, workspace=wsp)
    assert smr.get_device_error(wsp) == 0
    rep = check_route(ri, ids, wts, None)
    check_route_properties(ri, ids, wts)
    al = check_align(ids, 513, 128, srt, eids, npp)
    record("large_batch_M16384", rep, logits_out=False, npp=al.npp, block_size=128)
    print(f"large_batch: {rep}")


def test_large_batch_logits_every_tile(smr):
    """M=16384 with the logits output: every logit of two rows of each
    64-row tile (and the first and last tile whole) inside the accumulation
    bound, selection on them exact."""
    ri = inputs.large_batch()
    ids, wts, srt, eids, npp, lg = _route_align(smr, ri, 128)
    rng = np.random.default_rng(99)
    tiles = np.arange(0, ri.M, 64)
    rows = np.unique(np.concatenate([np.arange(0, 64), np.arange(ri.M - 64, ri.M),
                                     tiles + rng.integers(0, 64, tiles.size),
                                     tiles + rng.integers(0, 64, tiles.size)]))
    rep = check_route(ri, ids, wts, lg, rows=rows)
    check_align(ids, 513, 128, srt, eids, npp)
    record("large_batch_M16384_logits_sampled", rep, logits_out=True, npp=int(npp[0]), block_size=128)
    print(f"large_batch (logits, sampled): {rep}")


# ------------------------------------------------------------ edge cases --

@pytest.mark.parametrize("M,H,E,k,S", [
    (1, 8, 1, 1, 0),        # smallest problem
    (16, 4096, 512, 10, 1),  # largest small-M batch
    (5, 200, 37, 5, 1),      # H not a multiple of 64, odd E
    (7, 16384, 64, 8, 0),    # largest H, several passes per thread
    (2, 1024, 1024, 31, 1),  # largest E, widest row
    (17, 256, 64, 8, 1),     # smallest tcgen05 batch
    (130, 200, 96, 6, 1),    # two tiles, ragged tail, ragged K
    (300, 512, 512, 16, 0),  # k = 16 threshold classes
    (64, 128, 32, 32, 0),    # k = E, 32 classes
    (256, 2048, 256, 1, 1),  # k = 1
    # M > 16 outside the fused epilogue: logits-only tcgen05 launches + select
    (300, 512, 1024, 10, 1),   # the largest E: two 512-column launches
    (130, 200, 100, 8, 1),     # E not a multiple of 32, ragged K and tail
    (17, 64, 8, 4, 0),         # tiny E: one 32-column launch, 24 padded columns
    (1000, 1024, 600, 31, 1),  # a 512-column launch + an 88-column one, widest row
])
def test_shapes(smr, M, H, E, k, S):
    ri = inputs.make_route_inputs(M, H, E, k, S, seed=M * 1000 + E, shared_scale=0.75)
    _full_check(smr, ri, 64)


@pytest.mark.parametrize("M,H,E,k,S,zipf,launches", [
    (2049, 1024, 1000, 8, 1, 1.1, 2 + 1 + 3),  # logits in two launches, select, three align launches
    (16384, 4096, 1024, 10, 1, None, 2 + 1 + 3),
])
def test_generic_route_align(smr, M, H, E, k, S, zipf, launches):
    """M > 16 with E beyond the fused epilogue, through route_align as the
    benchmark calls it (no logits output): every row against the oracle."""
    ri = inputs.make_route_inputs(M, H, E, k, S, seed=M + E, zipf_s=zipf)
    rep, al, ids = _full_check(smr, ri, 128, with_logits=False, name=f"generic_M{M}_E{E}")
    assert smr.last_launch_count() == launches
    print(f"generic M={M} E={E}: {rep}")


@pytest.mark.parametrize("M,E,k,S,A", [
    (17, 64, 8, 1, 64),      # smallest tcgen05 batch
    (40, 256, 12, 1, 0),     # 520 slots, tier block size
    (64, 512, 10, 1, 128),   # 704 slots: the most the route's last CTA aligns
    (88, 128, 8, 0, 0),      # 704 slots at k = 8
])
def test_mid_m_route_align_is_one_launch(smr, M, E, k, S, A):
    """Mid M: the route's last CTA aligns all ids (the shared expert appended
    as expert E), so route_align is one launch; three calls in a row on one
    workspace each match the oracle and leave the ticket at zero."""
    ri = inputs.make_route_inputs(M, 1024, E, k, S, seed=900 + M)
    wsp = smr.Workspace()
    Aeff = A if A > 0 else oracle.select_block_size(M, k, E)
    for _ in range(3):
        ids, wts, srt, eids, npp, _ = _route_align(smr, ri, A, with_logits=False, workspace=wsp)
        assert smr.last_launch_count() == 1
        check_route(ri, ids, wts, None)
        check_align(ids, E + S, Aeff, srt, eids, npp)
    assert int(wsp.buf[12:16].view(torch.int32).item()) == 0  # the ticket
    assert smr.get_device_error(wsp) == 0


@pytest.mark.parametrize("M,H,E,k,S,zipf", [
    (1000, 1024, 512, 10, 1, None),  # 11000 slots: the route counts 16 tiles, the last 40 rows
    (777, 512, 256, 12, 0, 1.1),     # odd CTA count (7 tiles in 4 pairs), ragged tile, bias
    (2049, 256, 128, 8, 1, None),    # 33 count tiles, last one a single row
    (300, 512, 128, 8, 0, 1.1),      # 2400 slots, 5 count tiles
    (65, 1024, 512, 10, 1, None),    # 715 slots: just above the fused align, 2 count tiles
    (128, 1024, 128, 8, 0, None),    # the short prefill: 1024 slots, 2 count tiles
    (186, 1024, 512, 10, 1, 1.1),    # 2046 slots, a ragged count tile
])
def test_route_align_counts_from_route(smr, M, H, E, k, S, zipf):
    """route_align above the align fused into the route: the tcgen05 route writes each
    64-row tile's expert counts and the align scans and scatters from them."""
    ri = inputs.make_route_inputs(M, H, E, k, S, seed=M + E, zipf_s=zipf)
    assert M * (k + S) > 704  # above the align fused into the route
    _full_check(smr, ri, 128)
    assert smr.last_launch_count() == 3  # route + tile scan + tile scatter


def test_counted_align_after_other_calls_on_one_workspace(smr):
    """The counted align's tile arrays share the workspace with every other
    call's scratch (the logit rows of the generic route, the small route's
    tagged keys, the standalone align's tile arrays): any call sequence on one
    workspace gives the oracle's results, and the header's ticket and error
    word end at zero."""
    wsp = smr.Workspace()
    big = inputs.make_route_inputs(2049, 512, 256, 8, 1, seed=77)
    x, w, ws, b = _dev(big)
    ref = None
    for step in range(3):
        # something else writes where the group totals live
        if step == 0:
            gen = inputs.make_route_inputs(2049, 256, 1000, 8, 1, seed=78)  # generic: logit rows
            gx, gw, gws, gb = _dev(gen)
            smr.route_align(gx, gw, gws, gb, topk=8, block_size=64, workspace=wsp)
        elif step == 1:
            ids0 = torch.from_numpy(inputs.random_ids(3000, 9, 257, seed=5)).cuda()
            smr.align(ids0, 257, 16, workspace=wsp)  # standalone multi-tile align
        else:
            sm = inputs.make_route_inputs(16, 1024, 1024, 8, 1, seed=79)  # tagged keys
            sx, sw, sws, sb = _dev(sm)
            smr.route_align(sx, sw, sws, sb, topk=8, block_size=64, workspace=wsp)
        out = smr.route_align(x, w, ws, b, topk=8, block_size=128, workspace=wsp)
        torch.cuda.synchronize()
        assert smr.last_launch_count() == 3
        ids, wts, srt, eids, npp = (t.cpu().numpy() for t in out)
        check_route(big, ids, wts, None)
        check_align(ids, 257, 128, srt, eids, npp)
        n = int(npp[0])  # only the first npp (npp / A) entries are defined
        got = (ids.copy(), srt[:n].copy(), eids[: n // 128].copy(), npp.copy())
        if ref is None:
            ref = got
        for a, r in zip(got, ref):
            assert np.array_equal(a, r)
        hdr = wsp.buf[:32].view(torch.int32).cpu().numpy()
        assert hdr[1] == 0 and hdr[3] == 0  # error, ticket


@pytest.mark.parametrize("M,E,k", [(200, 128, 8), (300, 256, 10), (150, 64, 8), (40, 96, 12)])
def test_quad_threshold_integer_ties(smr, M, E, k):
    """Column halves of at most 128 experts take their threshold over
    4-column maxima: integer inputs (exact fp32 sums, many equal logits,
    k as large as the number of quads) must give the oracle's ids, weights
    and align outputs bit for bit."""
    ri = inputs.make_route_inputs(M, 256, E, k, 1, seed=40 + M + E, dist="int")
    rep, al, ids = _full_check(smr, ri, 64, exact=True)
    assert rep.exact_rows == rep.rows


@pytest.mark.parametrize("M", [4, 40])
def test_all_equal_logits_lowest_ids_win(smr, M):
    ri = inputs.make_route_inputs(M, 256, 128, 8, 1, seed=3)
    ri.w[:] = ri.w[0]  # every expert row identical: all logits tie
    ids, wts, srt, eids, npp, lg = _route_align(smr, ri, 64)
    assert np.all(ids[:, :8] == np.arange(8))
    assert np.all(wts[:, :8] == np.float32(1 / 8))
    check_route(ri, ids, wts, lg)


@pytest.mark.parametrize("M,E,k", [(4, 512, 10), (13, 1024, 31), (300, 512, 10)])
def test_top_logits_in_few_lanes(smr, M, E, k):
    """The largest logits all sit in experts e with e % 32 < 3 (a bias of
    +8 on them), so far more than 32 keys reach the k-th largest maximum of
    32 interleaved lanes: the selections' exact fallbacks must give the
    oracle's answer."""
    ri = inputs.make_route_inputs(M, 512, E, k, 1, seed=21 + M)
    ri.bias = np.where(np.arange(E) % 32 < 3, 8.0, 0.0).astype(np.float32)
    rep, al, ids = _full_check(smr, ri, 64)
    assert np.all(ids[:, :k] % 32 < 3)


@pytest.mark.parametrize("M,A", [(16, 8), (9, 5), (16, 16), (16, 17), (3, 3), (1, 1), (12, 2)])
def test_small_batch_block_sizes(smr, M, A):
    """Single-launch route+align with block sizes around M on a 64-expert
    gate (experts shared by several tokens): A >= M places each id from the
    per-expert token masks (one block per expert), A < M ranks the ids
    (experts, the shared one first of all, span several blocks)."""
    ri = inputs.make_route_inputs(M, 512, 64, 8, 1, seed=31 + M * 7 + A)
    rep, al, ids = _full_check(smr, ri, A)
    assert smr.last_launch_count() == 1


def test_bias_and_strided_hidden(smr):
    ri = inputs.make_route_inputs(40, 512, 128, 8, 1, seed=5, zipf_s=1.1)
    x, w, ws, b = _dev(ri)
    big = torch.zeros((40, 520), dtype=torch.bfloat16, device="cuda")
    big[:, :512] = x
    xs = big[:, :512]  # row stride 520
    logits = torch.empty((40, 128), dtype=torch.int16, device="cuda")
    ids, wts = smr.route(xs, w, ws, b, topk=8, logits_out=logits)
    torch.cuda.synchronize()
    check_route(ri, ids.cpu().numpy(), wts.cpu().numpy(), logits.cpu().numpy().view(np.uint16))


def test_graph_replay_matches_eager(smr):
    for M in (4, 300):
        ri = inputs.make_route_inputs(M, 1024, 128, 8, 1, seed=11 + M)
        x, w, ws, b = _dev(ri)
        A = 64
        wsp = smr.Workspace()
        eager = smr.route_align(x, w, ws, b, topk=8, block_size=A, workspace=wsp)
        torch.cuda.synchronize()
        eager = [t.clone() for t in eager]
        outs = [torch.empty_like(t) for t in eager]
        for t in outs:
            t.fill_(-5)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            smr.route_align(x, w, ws, b, topk=8, block_size=A, topk_ids=outs[0],
                            topk_weights=outs[1], sorted_token_ids=outs[2], expert_ids=outs[3],
                            num_tokens_post_padded=outs[4], workspace=wsp)
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            smr.route_align(x, w, ws, b, topk=8, block_size=A, topk_ids=outs[0],
                            topk_weights=outs[1], sorted_token_ids=outs[2], expert_ids=outs[3],
                            num_tokens_post_padded=outs[4], workspace=wsp)
        for _ in range(3):
            for t in outs:
                t.fill_(-5)
            g.replay()
            torch.cuda.synchronize()
            n = int(eager[4].item())
            assert torch.equal(outs[0], eager[0]) and torch.equal(outs[1], eager[1])
            assert int(outs[4].item()) == n
            assert torch.equal(outs[2][:n], eager[2][:n])
            assert torch.equal(outs[3][: n // A], eager[3][: n // A])
        assert smr.get_device_error(wsp) == 0


def test_workspace_reuse_is_deterministic(smr):
    ri = inputs.small_verify(8, variant=1)
    x, w, ws, b = _dev(ri)
    wsp = smr.Workspace()
    first = [t.clone() for t in smr.route_align(x, w, ws, b, topk=10, block_size=64, workspace=wsp)]
    for _ in range(5):
        again = smr.route_align(x, w, ws, b, topk=10, block_size=64, workspace=wsp)
        torch.cuda.synchronize()
        n = int(first[4].item())
        assert torch.equal(again[0], first[0]) and torch.equal(again[1], first[1])
        assert torch.equal(again[2][:n], first[2][:n])
    # the small route's call tag advanced once per call: 6 calls on a fresh
    # workspace (top bit set on every tag)
    tag = int(wsp.buf[8:12].view(torch.int32).item()) & 0xFFFFFFFF
    assert tag == 0x80000000 | 6
    assert smr.get_device_error(wsp) == 0


def test_back_to_back_small_calls_share_a_workspace(smr):
    """Consecutive single-launch calls on one stream and one workspace: each
    call may launch while the previous one's tail still runs (it streams its
    gate weights, then waits for that call before touching the workspace or
    the hidden states). Every call must give the result of an isolated call."""
    cases = [inputs.make_route_inputs(M, 1024, 256, 8, 1, seed=60 + M) for M in (4, 9, 1, 16)]
    dev = [_dev(ri) for ri in cases]
    ref = []
    for (x, w, ws, b) in dev:
        out = smr.route_align(x, w, ws, b, topk=8, block_size=64, workspace=smr.Workspace())
        torch.cuda.synchronize()
        ref.append([t.clone() for t in out])
    wsp = smr.Workspace()
    got = []
    for i in range(12):
        x, w, ws, b = dev[i % 4]
        got.append(smr.route_align(x, w, ws, b, topk=8, block_size=64, workspace=wsp))
    torch.cuda.synchronize()
    for i, out in enumerate(got):
        r = ref[i % 4]
        n = int(r[4].item())
        assert torch.equal(out[0], r[0]) and torch.equal(out[1], r[1])
        assert int(out[4].item()) == n
        assert torch.equal(out[2][:n], r[2][:n]) and torch.equal(out[3][: n // 64], r[3][: n // 64])
    assert smr.get_device_error(wsp) == 0


# ----------------------------------------------------------------- align --

@pytest.mark.parametrize("T,W,E_al,A,skew", [
    (0, 11, 513, 64, None),        # empty input
    (1, 1, 1, 1, None),
    (4, 11, 513, 64, None),
    (186, 11, 513, 64, 1.1),       # single CTA near its limit (2046 slots)
    (187, 11, 513, 128, None),     # just above: the three multi-CTA launches
    (700, 11, 513, 64, 1.1),       # 7700 slots, one tile
    (16384, 11, 513, 128, 1.1),    # the large batch's shape
    (2048, 8, 128, 128, 2.0),      # very hot experts
    (3000, 3, 7, 200, None),       # odd block size, few experts
    (9000, 1, 1025, 16, None),     # widest expert range
    (262147, 11, 513, 128, 1.1),   # 2.9M slots: tiles grow past 1024 slots, ragged last tile
])
def test_align_standalone(smr, T, W, E_al, A, skew):
    ids = inputs.random_ids(T, W, E_al, seed=T + W + A, skew=skew) if T else np.zeros((0, W), np.int32)
    dids = torch.from_numpy(ids).cuda()
    srt, eids, npp = smr.align(dids, E_al, A)
    torch.cuda.synchronize()
    check_align(ids, E_al, A, srt.cpu().numpy(), eids.cpu().numpy(), npp.cpu().numpy())
    assert smr.last_launch_count() == (1 if T * W <= 2048 else 3)


def test_align_reused_workspace_back_to_back(smr):
    """Consecutive multi-tile aligns on one workspace and stream, alternating
    two id sets: each kernel may launch before its predecessor finishes, so
    what another kernel writes must be read through L2, never from a stale
    line of an earlier call on the same SM. Every result matches the oracle."""
    sets = [inputs.random_ids(60000, 11, 513, seed=s, skew=1.1) for s in (5, 6)]
    dids = [torch.from_numpy(i).cuda() for i in sets]
    wsp = smr.Workspace()
    outs = [smr.align(dids[i % 2], 513, 128, workspace=wsp) for i in range(6)]
    torch.cuda.synchronize()
    for i, (srt, eids, npp) in enumerate(outs):
        check_align(sets[i % 2], 513, 128, srt.cpu().numpy(), eids.cpu().numpy(), npp.cpu().numpy())
    assert smr.get_device_error(wsp) == 0


def test_route_align_reused_workspace_back_to_back(smr):
    """tcgen05 route + two-launch align, four calls on one workspace and
    stream with alternating inputs: each matches an isolated call."""
    cases = [inputs.make_route_inputs(2049, 512, 256, 8, 1, seed=s) for s in (71, 72)]
    dev = [_dev(ri) for ri in cases]
    ref = []
    for (x, w, ws, b) in dev:
        out = smr.route_align(x, w, ws, b, topk=8, block_size=128, workspace=smr.Workspace())
        torch.cuda.synchronize()
        ref.append([t.clone() for t in out])
    wsp = smr.Workspace()
    got = [smr.route_align(*dev[i % 2], topk=8, block_size=128, workspace=wsp) for i in range(4)]
    torch.cuda.synchronize()
    for i, out in enumerate(got):
        r = ref[i % 2]
        n = int(r[4].item())
        assert torch.equal(out[0], r[0]) and torch.equal(out[1], r[1])
        assert int(out[4].item()) == n
        assert torch.equal(out[2][:n], r[2][:n]) and torch.equal(out[3][: n // 128], r[3][: n // 128])
    assert smr.get_device_error(wsp) == 0


def test_align_bad_id_sets_error_bit(smr):
    ids = inputs.random_ids(20, 4, 16, seed=1)
    ids[3, 2] = 16  # out of range
    wsp = smr.Workspace()
    dids = torch.from_numpy(ids).cuda()
    smr.align(dids, 16, 64, workspace=wsp)
    assert smr.get_device_error(wsp) & smr.ERR_BAD_ID
    smr.clear_device_error(wsp)
    assert smr.get_device_error(wsp) == 0
