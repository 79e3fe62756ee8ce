"""Failure detection without a GPU fault. A test hook makes one bounded wait
of a kernel wait for something nothing provides (a call tag no row group
writes; a barrier nothing arrives on), with a short limit. The kernel must
return, set bit 1 (wait timeout) of the sticky error word, and leave the
workspace fit for the next call, which must match the oracle. Needs a GB300.
"""
from __future__ import annotations

import numpy as np
import pytest

from moe_router_top_gb300 import inputs

from _parity import check_align, check_route

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def smr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import moe_router_top_gb300 as m
    yield m
    m.test_force_wait_timeout(m.STALL_NONE)


def _dev(ri):
    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return bf(ri.x), bf(ri.w), bf(ri.ws)


def test_small_tail_wait_runs_out(smr):
    ri = inputs.make_route_inputs(4, 1024, 128, 8, 1, seed=91)
    x, w, ws = _dev(ri)
    wsp = smr.Workspace()
    smr.route_align(x, w, ws, topk=8, block_size=64, workspace=wsp)  # a normal call first
    assert smr.get_device_error(wsp) == 0
    try:
        smr.test_force_wait_timeout(smr.STALL_SMALL_TAIL, 64)
        smr.route_align(x, w, ws, topk=8, block_size=64, workspace=wsp)
        torch.cuda.synchronize()  # the kernel returned
    finally:
        smr.test_force_wait_timeout(smr.STALL_NONE)
    assert smr.get_device_error(wsp) & smr.ERR_WAIT_TIMEOUT
    smr.clear_device_error(wsp)
    # the next call on the same workspace is correct
    ids, wts, srt, eids, npp = smr.route_align(x, w, ws, topk=8, block_size=64, workspace=wsp)
    torch.cuda.synchronize()
    assert smr.get_device_error(wsp) == 0
    ids, wts = ids.cpu().numpy(), wts.cpu().numpy()
    check_route(ri, ids, wts, None)
    check_align(ids, 129, 64, srt.cpu().numpy(), eids.cpu().numpy(), npp.cpu().numpy())


def test_tcgen05_merge_wait_runs_out(smr):
    ri = inputs.make_route_inputs(300, 512, 256, 8, 1, seed=92)
    x, w, ws = _dev(ri)
    wsp = smr.Workspace()
    ids = torch.full((300, 9), -7, dtype=torch.int32, device="cuda")
    wts = torch.full((300, 9), -7.0, dtype=torch.float32, device="cuda")
    try:
        smr.test_force_wait_timeout(smr.STALL_TC_MERGE, 20000)  # SM cycles
        smr.route(x, w, ws, topk=8, topk_ids=ids, topk_weights=wts, workspace=wsp)
        torch.cuda.synchronize()  # the kernel returned
    finally:
        smr.test_force_wait_timeout(smr.STALL_NONE)
    assert smr.get_device_error(wsp) & smr.ERR_WAIT_TIMEOUT
    # a route whose wait ran out writes no outputs
    assert bool(torch.all(ids == -7).item()) and bool(torch.all(wts == -7.0).item())
    smr.clear_device_error(wsp)
    smr.route(x, w, ws, topk=8, topk_ids=ids, topk_weights=wts, workspace=wsp)
    torch.cuda.synchronize()
    assert smr.get_device_error(wsp) == 0
    check_route(ri, ids.cpu().numpy(), wts.cpu().numpy(), None)
