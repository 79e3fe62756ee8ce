"""GPU parity of the consumer expert GEMM (the align's consumer, with the
num_tokens_post_padded early exit) against the oracle's per-slot definition:
every output within the fp32 accumulation bound of the exact sum, at both
block sizes of the M-aware tier. Needs a GB300."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from moe_router_top_gb300 import inputs

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


@pytest.mark.parametrize("M,H,E,k,S,N,A,zipf", [
    (4, 4096, 512, 10, 1, 256, 64, None),   # verify-sized: every expert one partly padded block
    (300, 512, 64, 8, 1, 384, 64, 1.1),     # M = 64 tiles, 128-column N tiles, skewed
    (300, 512, 64, 8, 1, 512, 128, 1.1),    # M = 128 tiles, 256-column N tiles
    (1000, 256, 128, 8, 0, 128, 128, 2.0),  # hot experts over many blocks
])
def test_expert_gemm_matches_oracle(smr, M, H, E, k, S, N, A, zipf):
    ri = inputs.make_route_inputs(M, H, E, k, S, seed=1000 + M + A, zipf_s=zipf)
    x, w = _bf16(ri.x), _bf16(ri.w)
    ws = _bf16(ri.ws) if S else None
    b = torch.from_numpy(ri.bias).cuda() if ri.bias is not None else None
    ids, wts, srt, eids, npp = smr.route_align(x, w, ws, b, topk=k, block_size=A)
    rng = np.random.default_rng(2000 + M)
    ew = inputs.f32_to_bf16_bits(rng.normal(0, 0.05, (E + S, N, H)).astype(np.float32))
    out = torch.full((M * (k + S), N), float("nan"), dtype=torch.float32, device="cuda")
    wsp = smr.Workspace()
    smr.expert_gemm(x, _bf16(ew), srt, eids, npp, width=k + S, block_size=A, out=out, workspace=wsp)
    torch.cuda.synchronize()
    assert smr.get_device_error(wsp) == 0 and smr.last_launch_count() == 1
    got = out.cpu().numpy().astype(np.float64)
    ref, ad = oracle.expert_gemm(ri.x, ids.cpu().numpy(), ew)
    bound = 2.0 * (H // 16 + 32) * 2.0 ** -24 * ad  # fp32: one update per K = 16 instruction
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), "a routed slot's row was not written"
    assert np.all(err <= bound), f"max error / bound {np.max(err / np.maximum(bound, 1e-300)):.3g}"
