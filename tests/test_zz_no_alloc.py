"""The no-allocation route+align entry point (smr_route_align_static).

It serves callers that cannot allocate device memory on their launch path:
instead of a caller workspace it uses the library's fixed device scratch
array. Its results must equal those of smr_route_align with a workspace, on
two calls in a row (the second call reuses the array the first one left
behind). Collected last on purpose, so that a stop at the first failure has
already run every other test; it passes alone in a fresh process as well.
"""
from __future__ import annotations

import numpy as np
import pytest

from moe_router_top_gb300 import inputs

from _parity import check_align, check_route, weights_close

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


CASES = [
    # verify-sized batch with the shared expert, and a biased 128-expert batch
    inputs.make_route_inputs(4, 4096, 512, 10, 1, seed=401, block_size=64),
    inputs.make_route_inputs(16, 2048, 128, 8, 0, seed=402, zipf_s=1.1, block_size=0),
]


@pytest.mark.parametrize("ri", CASES, ids=["M4_E512_shared", "M16_E128_bias"])
def test_static_scratch_matches_workspace_path(smr, ri):
    x, w = _bf16(ri.x), _bf16(ri.w)
    ws = _bf16(ri.ws) if ri.ws is not None else None
    b = torch.from_numpy(ri.bias).cuda() if ri.bias is not None else None
    ref = smr.route_align(x, w, ws, b, topk=ri.topk, block_size=ri.block_size,
                          workspace=smr.Workspace())
    torch.cuda.synchronize()
    ref = [t.cpu().numpy() for t in ref]
    A = ri.block_size or smr.select_block_size(ri.M, ri.topk, ri.E)
    n = int(ref[4][0])
    for _ in range(2):  # two calls in a row on the shared array
        got = smr.route_align_static(x, w, ws, b, topk=ri.topk, block_size=ri.block_size)
        torch.cuda.synchronize()
        ids, wts, srt, eids, npp = (t.cpu().numpy() for t in got)
        assert np.array_equal(ids, ref[0])
        assert weights_close(wts, ref[1]).all()
        assert int(npp[0]) == n
        assert np.array_equal(srt[:n], ref[2][:n])
        assert np.array_equal(eids[: n // A], ref[3][: n // A])
        # and against the oracle itself
        check_route(ri, ids, wts, None)
        check_align(ids, ri.num_experts_align, A, srt, eids, npp)
    assert smr.last_launch_count() == 1
    # the fixed array's sticky error word is readable and clear
    assert smr.get_static_device_error() == 0
    smr.clear_static_device_error()
    assert smr.get_static_device_error() == 0


def test_static_scratch_refuses_large_batches(smr):
    ri = inputs.make_route_inputs(17, 256, 64, 4, 1, seed=403)
    with pytest.raises(smr.SmrUnsupported, match="1 <= M <= 16"):
        smr.route_align_static(_bf16(ri.x), _bf16(ri.w), _bf16(ri.ws), topk=4, block_size=64)
