"""GPU parity of the hidden states quantised in the route's launch (E4M3,
one scale per 128 values) against the oracle: codes and scales bit-exact on
every path (single launch, fused tcgen05 route, logits-only launches), with
the routing outputs unchanged. Needs a GB300."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from moe_router_top_gb300 import inputs

from _parity import check_route

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


@pytest.mark.parametrize("M,H,E,k,S", [
    (4, 4096, 512, 10, 1),      # single launch, verify-sized
    (16, 1024, 128, 8, 0),      # single launch, no shared gate
    (300, 4096, 512, 10, 1),    # fused tcgen05 route, ragged tail
    (200, 256, 64, 4, 0),       # fused tcgen05 route, two blocks per row, no shared gate
    (130, 512, 1000, 8, 1),     # logits-only launches (the first quantises)
    (16384, 4096, 512, 10, 1),  # the large batch
])
def test_hidden_fp8_matches_oracle(smr, M, H, E, k, S):
    ri = inputs.make_route_inputs(M, H, E, k, S, seed=800 + M)
    ri.x[0, :128] = 0                          # a block of zeros
    ri.x[min(1, M - 1), 128:256] = 0x8000      # a block of negative zeros
    x, w = _bf16(ri.x), _bf16(ri.w)
    ws = _bf16(ri.ws) if S else None
    q = torch.full((M, H), 0xAA, dtype=torch.uint8, device="cuda")
    sc = torch.full((M, H // 128), -1.0, dtype=torch.float32, device="cuda")
    ids, wts, *_ = smr.route_align(x, w, ws, topk=k, block_size=128, hidden_fp8=q, hidden_scales=sc)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_fp8(ri.x)
    gq, gs = q.cpu().numpy(), sc.cpu().numpy()
    bad = np.nonzero(gq != rq)
    assert bad[0].size == 0, f"{bad[0].size} codes differ, e.g. row {bad[0][0]} col {bad[1][0]}: {gq[bad][0]:#x} vs {rq[bad][0]:#x}"
    assert np.array_equal(gs.view(np.uint32), rs.view(np.uint32))
    rows = None if M <= 4096 else np.arange(0, M, 13)
    check_route(ri, ids.cpu().numpy(), wts.cpu().numpy(), None, rows=rows)


def test_hidden_fp8_refused_without_whole_blocks(smr):
    ri = inputs.make_route_inputs(4, 200, 64, 4, 1, seed=801)
    with pytest.raises(smr.SmrError, match="H % 128"):
        smr.route(_bf16(ri.x), _bf16(ri.w), _bf16(ri.ws), topk=4,
                  hidden_fp8=torch.empty((4, 200), dtype=torch.uint8, device="cuda"),
                  hidden_scales=torch.empty((4, 1), dtype=torch.float32, device="cuda"))
