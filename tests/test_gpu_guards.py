"""Guard regions around every output buffer, and one workspace shared by all
paths. Needs a GB300.

compute-sanitizer is not available on this machine, so each output of the
C ABI is handed over as the interior of a larger buffer whose margins hold a
canary pattern: after the call every margin must be intact (no write lands
outside the caller's arrays) and the interior must still match the oracle.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from moe_router_top_gb300 import inputs

from _parity import check_align, check_route

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

G = 256  # canary words on each side (1 KB: keeps the interiors 16-byte aligned)
CANARY = {torch.int32: -0x21524111, torch.float32: -1234.5, torch.int16: -12345}


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


class Guarded:
    """A buffer of n elements (shaped `shape`) between two canary margins."""

    def __init__(self, shape, dtype):
        self.n = int(np.prod(shape))
        self.dtype = dtype
        self.buf = torch.full((self.n + 2 * G,), CANARY[dtype], dtype=dtype, device="cuda")
        self.view = self.buf[G:G + self.n].view(*shape)

    def intact(self) -> bool:
        c = CANARY[self.dtype]
        return bool(torch.all(self.buf[:G] == c).item()) and bool(torch.all(self.buf[G + self.n:] == c).item())


@pytest.mark.parametrize("M,H,E,k,S,A", [
    (4, 4096, 512, 10, 1, 64),    # single launch, bulk-copied align
    (16, 2048, 128, 8, 0, 0),     # single launch, tier block size
    (9, 512, 64, 8, 1, 5),        # single launch, A < M: ranked align, direct stores
    (300, 512, 256, 8, 1, 64),    # tcgen05 route + one-CTA align
    (2049, 256, 128, 8, 1, 128),  # tcgen05 route + counted multi-tile align
    (300, 512, 1000, 10, 1, 64),  # logits-only tcgen05 launches + select + one-CTA align
])
def test_route_align_writes_stay_inside_outputs(smr, M, H, E, k, S, A):
    ri = inputs.make_route_inputs(M, H, E, k, S, seed=500 + M + E)
    x, w = _bf16(ri.x), _bf16(ri.w)
    ws = _bf16(ri.ws) if ri.ws is not None else None
    width = k + S
    Aeff = A if A > 0 else oracle.select_block_size(M, k, E)
    cap = smr.align_capacity(M * width, E + S, Aeff)
    g = {
        "ids": Guarded((M, width), torch.int32),
        "wts": Guarded((M, width), torch.float32),
        "logits": Guarded((M, E), torch.int16),
        "srt": Guarded((cap,), torch.int32),
        "eids": Guarded(((cap + Aeff - 1) // Aeff,), torch.int32),
        "npp": Guarded((1,), torch.int32),
    }
    wsp = smr.Workspace()
    smr.route_align(x, w, ws, topk=k, block_size=A, logits_out=g["logits"].view,
                    topk_ids=g["ids"].view, topk_weights=g["wts"].view,
                    sorted_token_ids=g["srt"].view, expert_ids=g["eids"].view,
                    num_tokens_post_padded=g["npp"].view, workspace=wsp)
    torch.cuda.synchronize()
    for name, gb in g.items():
        assert gb.intact(), f"{name}: a write landed outside the output array"
    ids = g["ids"].view.cpu().numpy()
    check_route(ri, ids, g["wts"].view.cpu().numpy(), g["logits"].view.cpu().numpy().view(np.uint16))
    check_align(ids, E + S, Aeff, g["srt"].view.cpu().numpy(), g["eids"].view.cpu().numpy(),
                g["npp"].view.cpu().numpy())
    assert smr.get_device_error(wsp) == 0


@pytest.mark.parametrize("T,W,E_al,A", [(700, 11, 513, 64), (30000, 11, 513, 128), (3000, 3, 7, 200)])
def test_align_writes_stay_inside_outputs(smr, T, W, E_al, A):
    ids = inputs.random_ids(T, W, E_al, seed=T + A, skew=1.1)
    cap = smr.align_capacity(T * W, E_al, A)
    srt = Guarded((cap,), torch.int32)
    eids = Guarded(((cap + A - 1) // A,), torch.int32)
    npp = Guarded((1,), torch.int32)
    smr.align(torch.from_numpy(ids).cuda(), E_al, A, sorted_token_ids=srt.view,
              expert_ids=eids.view, num_tokens_post_padded=npp.view)
    torch.cuda.synchronize()
    assert srt.intact() and eids.intact() and npp.intact()
    check_align(ids, E_al, A, srt.view.cpu().numpy(), eids.view.cpu().numpy(), npp.view.cpu().numpy())


def test_one_workspace_for_every_path(smr):
    """A multi-tile align leaves nonnegative int32 in the workspace, a tcgen05
    route_align its tile counts; the small route's tagged key words must
    never take either for the current call's keys. Every call, in any
    order on one workspace, matches a call on a fresh workspace."""
    small = inputs.make_route_inputs(4, 1024, 128, 8, 1, seed=601)
    big = inputs.make_route_inputs(2049, 256, 128, 8, 1, seed=602)
    ids_a = inputs.random_ids(30000, 11, 513, seed=603, skew=1.1)

    def run_small(wsp):
        return smr.route_align(_bf16(small.x), _bf16(small.w), _bf16(small.ws), topk=8,
                               block_size=64, workspace=wsp)

    def run_big(wsp):
        return smr.route_align(_bf16(big.x), _bf16(big.w), _bf16(big.ws), topk=8,
                               block_size=128, workspace=wsp)

    def run_align(wsp):
        return smr.align(torch.from_numpy(ids_a).cuda(), 513, 128, workspace=wsp)

    def same(a, b, A):
        a = [t.cpu() for t in a]
        b = [t.cpu() for t in b]
        n = int(a[-1].item())
        assert int(b[-1].item()) == n
        for x, y in zip(a[:-3], b[:-3]):  # routed ids and weights
            assert torch.equal(x, y)
        assert torch.equal(a[-3][:n], b[-3][:n]) and torch.equal(a[-2][: n // A], b[-2][: n // A])

    ref = {"s": run_small(smr.Workspace()), "b": run_big(smr.Workspace()), "a": run_align(smr.Workspace())}
    torch.cuda.synchronize()
    wsp = smr.Workspace()
    for kind in ("a", "s", "b", "s", "a", "s"):
        got = {"s": run_small, "b": run_big, "a": run_align}[kind](wsp)
        torch.cuda.synchronize()
        same(got, ref[kind], 64 if kind == "s" else 128)
    assert smr.get_device_error(wsp) == 0
