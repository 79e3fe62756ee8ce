"""GPU parity of the routing variants against the oracle: weights without
renormalisation (the E-expert softmax at the top-k ids), a bf16-rounded
shared logit, and the EPLB logical->physical remap inside the align. Both
route paths (single launch M <= 16, tcgen05 M > 16) and every align path
(one CTA, multi-tile). Needs a GB300."""
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
    ws = _bf16(ri.ws) if ri.ws is not None else None
    b = torch.from_numpy(ri.bias).cuda() if ri.bias is not None else None
    return _bf16(ri.x), _bf16(ri.w), ws, b


VARIANT_SHAPES = [
    (4, 4096, 512, 10, 1, None),     # single launch, verify-sized
    (13, 1024, 1024, 31, 1, None),   # single launch, widest row
    (300, 512, 256, 8, 1, None),     # tcgen05, two tiles with a ragged tail
    (2049, 2048, 128, 8, 0, 1.1),    # tcgen05, skewed, counted multi-tile align
    (16384, 4096, 512, 10, 1, None), # the large batch
]


@pytest.mark.parametrize("with_logits", [False, True], ids=["no_logits", "logits_out"])
@pytest.mark.parametrize("M,H,E,k,S,zipf", VARIANT_SHAPES)
def test_no_renormalisation(smr, M, H, E, k, S, zipf, with_logits):
    ri = inputs.make_route_inputs(M, H, E, k, S, seed=500 + M, zipf_s=zipf, renormalize=False)
    x, w, ws, b = _dev(ri)
    logits = torch.empty((M, E), dtype=torch.int16, device="cuda") if with_logits else None
    ids, wts, srt, eids, npp = smr.route_align(x, w, ws, b, topk=k, block_size=128,
                                                renormalize=False, logits_out=logits)
    torch.cuda.synchronize()
    ids, wts = ids.cpu().numpy(), wts.cpu().numpy()
    lg = logits.cpu().numpy().view(np.uint16) if with_logits else None
    rows = None if M <= 4096 else np.arange(0, M, 7)
    rep = check_route(ri, ids, wts, lg, rows=rows)
    check_route_properties(ri, ids, wts)
    assert np.all(wts[:, :k].astype(np.float64).sum(axis=1) < 1.0)
    check_align(ids, E + S, 128, srt.cpu().numpy(), eids.cpu().numpy(), npp.cpu().numpy())
    record(f"no_renorm_M{M}_E{E}" + ("_logits" if with_logits else ""), rep, logits_out=with_logits)


@pytest.mark.parametrize("M", [1, 3, 8])
def test_no_renormalisation_tie_stress_exact(smr, M):
    """Integer inputs (exact fp32 accumulation): ids bit-exact, weights of
    the E-expert softmax within 2e-6 of the oracle's on every row."""
    ri = inputs.tie_stress(M)
    ri.renormalize = False
    x, w, ws, b = _dev(ri)
    ids, wts = smr.route(x, w, ws, topk=10, renormalize=False)
    torch.cuda.synchronize()
    rep = check_route(ri, ids.cpu().numpy(), wts.cpu().numpy(), None, exact_logits=True)
    assert rep.exact_rows == rep.rows


@pytest.mark.parametrize("M,H,E,k", [(4, 4096, 512, 10), (16, 512, 64, 8), (300, 512, 256, 8),
                                     (16384, 4096, 512, 10)])
def test_shared_logit_rounded_to_bf16(smr, M, H, E, k):
    ri = inputs.make_route_inputs(M, H, E, k, 1, seed=600 + M, shared_scale=0.75, shared_bf16=True)
    x, w, ws, b = _dev(ri)
    ids, wts = smr.route(x, w, ws, topk=k, shared_scale=0.75, shared_logit_bf16=True)
    torch.cuda.synchronize()
    rows = None if M <= 4096 else np.arange(0, M, 7)
    rep = check_route(ri, ids.cpu().numpy(), wts.cpu().numpy(), None, rows=rows)
    record(f"shared_bf16_M{M}", rep, logits_out=False)
    # the flag is not a no-op on these inputs
    ref0 = oracle.route(ri.x[:4], ri.w, ri.ws, None, k, 0.75)
    assert not np.array_equal(ref0.w[:, k], wts.cpu().numpy()[:4, k])


def _eplb_case(E_al, R, P, seed):
    emap, cnt = inputs.random_eplb_map(E_al, R, P, seed=seed)
    return emap, cnt, torch.from_numpy(emap).cuda(), torch.from_numpy(cnt).cuda()


@pytest.mark.parametrize("T,W,E_al,R,P,A,skew", [
    (5, 11, 513, 3, 700, 64, None),        # one align CTA
    (700, 11, 513, 4, 1025, 64, 1.1),      # one CTA near its limit, hot experts replicated
    (16384, 11, 513, 2, 800, 128, 1.1),    # multi-tile, the large batch's shape
    (3000, 3, 7, 8, 40, 16, 2.0),          # few experts, many replicas
])
def test_align_eplb(smr, T, W, E_al, R, P, A, skew):
    ids = inputs.random_ids(T, W, E_al, seed=T + R, skew=skew)
    emap, cnt, demap, dcnt = _eplb_case(E_al, R, P, seed=T * 3 + P)
    wsp = smr.Workspace()
    srt, eids, npp = smr.align(torch.from_numpy(ids).cuda(), E_al, A, eplb_map=demap,
                               eplb_count=dcnt, num_physical=P, workspace=wsp)
    torch.cuda.synchronize()
    ref = oracle.align_eplb(ids, E_al, emap, cnt, P, A)
    n = int(npp.item())
    assert n == ref.npp
    assert np.array_equal(srt.cpu().numpy()[:n], ref.sorted_ids)
    assert np.array_equal(eids.cpu().numpy()[: n // A], ref.expert_ids)
    assert smr.get_device_error(wsp) == 0


@pytest.mark.parametrize("M,H,E,k,S,R,P", [
    (4, 4096, 512, 10, 1, 2, 700),     # small batch: route launch + one align launch
    (2049, 512, 128, 8, 1, 3, 300),    # tcgen05 route + three align launches
])
def test_route_align_eplb(smr, M, H, E, k, S, R, P):
    ri = inputs.make_route_inputs(M, H, E, k, S, seed=700 + M)
    x, w, ws, b = _dev(ri)
    emap, cnt, demap, dcnt = _eplb_case(E + S, R, P, seed=M)
    A = 64
    ids, wts, srt, eids, npp = smr.route_align(x, w, ws, b, topk=k, block_size=A, eplb_map=demap,
                                                eplb_count=dcnt, num_physical=P)
    torch.cuda.synchronize()
    launches = smr.last_launch_count()
    assert launches == 1 + (1 if M * (k + S) <= 2048 else 3)
    ids = ids.cpu().numpy()
    check_route(ri, ids, wts.cpu().numpy(), None)
    ref = oracle.align_eplb(ids, E + S, emap, cnt, P, A)
    n = int(npp.item())
    assert n == ref.npp
    assert np.array_equal(srt.cpu().numpy()[:n], ref.sorted_ids)
    assert np.array_equal(eids.cpu().numpy()[: n // A], ref.expert_ids)


def test_align_eplb_bad_physical_id_sets_error_bit(smr):
    ids = inputs.random_ids(20, 4, 16, seed=2)
    emap, cnt = inputs.random_eplb_map(16, 2, 40, seed=3)
    emap[int(ids[0, 0]), 0] = 40  # a physical id out of range
    wsp = smr.Workspace()
    smr.align(torch.from_numpy(ids).cuda(), 16, 8, eplb_map=torch.from_numpy(emap).cuda(),
              eplb_count=torch.from_numpy(cnt).cuda(), num_physical=40, workspace=wsp)
    assert smr.get_device_error(wsp) & smr.ERR_BAD_ID
