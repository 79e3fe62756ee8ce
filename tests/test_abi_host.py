"""Host-side tests of the C ABI (no GPU needed): the library loads and exports
every function include/smr.h declares; refusals list every reason and happen
before any device work; workspace sizes, the tier and the capacity helpers.
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import oracle
from moe_router_top_gb300 import _lib
from moe_router_top_gb300._lib import AlignArgs, RouteArgs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from moe_router_top_gb300 import build
    build.build()
    return _lib.load()


def _header_functions():
    text = open(os.path.join(ROOT, "include", "smr.h")).read()
    return sorted(set(re.findall(r"SMR_API\s+[\w\s\*]+?\b(smr_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    declared = _header_functions()
    assert len(declared) >= 14
    assert sorted(_lib.EXPORTED) == declared
    for name in declared:
        assert hasattr(lib, name), name


def test_struct_layouts_match_header(lib):
    # field order and sizes as declared in include/smr.h (LP64)
    assert ctypes.sizeof(RouteArgs) == 7 * 4 + 4 + 8 * 8 + 8 + 2 * 8  # + shared_logit_bf16, e4m3 outputs
    assert RouteArgs.hidden.offset == 32
    assert RouteArgs.shared_logit_bf16.offset == 96 and RouteArgs.hidden_fp8.offset == 104
    assert ctypes.sizeof(AlignArgs) == 8 + 6 * 4 + 5 * 8 + 2 * 8 + 2 * 4
    assert AlignArgs.sorted_token_ids.offset == 32
    assert AlignArgs.eplb_map.offset == 72 and AlignArgs.num_physical.offset == 92


def test_version_and_status_strings(lib):
    assert lib.smr_version() == 0x000200
    assert lib.smr_status_string(0) == b"SMR_OK"
    assert lib.smr_status_string(2) == b"SMR_ERR_UNSUPPORTED"


def _good_route(M=4, H=4096, E=512, k=10, S=1):
    a = RouteArgs()
    a.M, a.H, a.E, a.topk, a.has_shared = M, H, E, k, S
    a.shared_scale = 1.0
    a.renormalize = 1
    a.hidden = 0x10000
    a.ld_hidden = H
    a.gate_w = 0x20000
    a.shared_w = 0x30000 if S else None
    a.bias = None
    a.topk_ids = 0x40000
    a.topk_weights = 0x50000
    return a


def test_route_refusal_lists_every_reason(lib):
    a = _good_route()
    a.H = 4100          # not a multiple of 8
    a.hidden = 0x10004  # misaligned
    a.shared_w = None   # has_shared but NULL
    a.topk_ids = None
    st = lib.smr_route(ctypes.byref(a), None, 0, None)
    assert st == _lib.SMR_ERR_INVALID_ARG
    msg = lib.smr_last_error().decode()
    for frag in ("H must be a multiple of 8", "hidden must be 16-byte aligned",
                 "shared_w is NULL", "topk_ids is NULL"):
        assert frag in msg, msg
    assert lib.smr_last_launch_count() == 0


def test_route_variant_flags_checked(lib):
    a = _good_route()
    a.renormalize = 2
    a.shared_logit_bf16 = 3
    assert lib.smr_route(ctypes.byref(a), None, 0, None) == _lib.SMR_ERR_INVALID_ARG
    msg = lib.smr_last_error().decode()
    assert "renormalize must be 0 or 1" in msg and "shared_logit_bf16 must be 0 or 1" in msg
    a.renormalize, a.shared_logit_bf16 = 0, 1  # both variants are implemented
    assert lib.smr_route(ctypes.byref(a), None, 0, None) == _lib.SMR_ERR_WORKSPACE


def test_route_unsupported_contract(lib):
    for E in (500, 1024, 40):         # outside the fused epilogue: logits + select, admitted
        a = _good_route(M=64, E=E)
        need = lib.smr_route_workspace_size(ctypes.byref(a))
        ld = (E + 31) // 32 * 32      # bf16 logit rows + fp32 shared logits in the workspace
        assert need == 256 + ((64 * ld * 2 + 255) // 256) * 256 + 256
        assert lib.smr_route(ctypes.byref(a), None, 0, None) == _lib.SMR_ERR_WORKSPACE
    a = _good_route(M=64, E=512)      # fused epilogue: no workspace beyond the header
    assert lib.smr_route_workspace_size(ctypes.byref(a)) == 256
    a = _good_route(k=32, S=1, E=64)  # width 33 > 32
    assert lib.smr_route(ctypes.byref(a), None, 0, None) == _lib.SMR_ERR_UNSUPPORTED


def test_route_workspace_checked_before_device(lib):
    a = _good_route()
    need = lib.smr_route_workspace_size(ctypes.byref(a))
    assert need == 256 + ((4 * 512 * 8 + 255) // 256) * 256  # header + [M][E] tagged 8-byte keys
    assert lib.smr_route(ctypes.byref(a), None, 0, None) == _lib.SMR_ERR_WORKSPACE
    assert lib.smr_route(ctypes.byref(a), 0x100080, need, None) == _lib.SMR_ERR_WORKSPACE  # misaligned
    assert lib.smr_route(ctypes.byref(a), 0x100000, need - 1, None) == _lib.SMR_ERR_WORKSPACE
    big = _good_route(M=16384)
    assert lib.smr_route_workspace_size(ctypes.byref(big)) == 256  # tcgen05 path keeps no scratch


def test_route_m0_is_a_no_op(lib):
    a = _good_route(M=0)
    a.hidden = a.gate_w = a.shared_w = a.topk_ids = a.topk_weights = None
    assert lib.smr_route(ctypes.byref(a), None, 0, None) == _lib.SMR_OK
    assert lib.smr_last_launch_count() == 0


def _good_align(T=4, W=11, E_al=513, A=64):
    a = AlignArgs()
    a.topk_ids = 0x10000
    a.num_tokens, a.width, a.num_experts = T, W, E_al
    a.routed_topk, a.routed_experts = W - 1, E_al - 1
    a.block_size = A
    cap = T * W + E_al * (max(A, 64) - 1) if A else T * W + E_al * 127
    a.sorted_token_ids = 0x20000
    a.sorted_cap = cap
    a.expert_ids = 0x30000
    a.expert_cap = cap
    a.num_tokens_post_padded = 0x40000
    return a


def test_align_refusals(lib):
    a = _good_align()
    a.sorted_cap = 10
    a.num_tokens_post_padded = None
    assert lib.smr_align(ctypes.byref(a), None, 0, None) == _lib.SMR_ERR_INVALID_ARG
    msg = lib.smr_last_error().decode()
    assert "sorted_cap 10 < required 32363" in msg and "num_tokens_post_padded is NULL" in msg
    a = _good_align(A=0)
    a.routed_topk = 0
    assert lib.smr_align(ctypes.byref(a), None, 0, None) == _lib.SMR_ERR_INVALID_ARG
    assert "routed_topk" in lib.smr_last_error().decode()


def test_align_workspace_sizes(lib):
    a = _good_align(T=4)
    assert lib.smr_align_workspace_size(ctypes.byref(a)) == 256          # one CTA, no scratch
    a = _good_align(T=16384, A=128)
    # tiles of 1024 slots (at most 2048 tiles): [tiles][E_al] counts and
    # starts, [E_al] totals
    ntiles = (16384 * 11 + 1023) // 1024
    words = 2 * ntiles * 513 + 513
    assert lib.smr_align_workspace_size(ctypes.byref(a)) == 256 + ((words * 4 + 255) // 256) * 256
    a = _good_align(T=1 << 22, W=64, A=128)  # 2^28 slots: tiles grow to keep 2048 of them
    tile = -(-(1 << 28) // 2048)
    tile = -(-tile // 1024) * 1024
    ntiles = -(-(1 << 28) // tile)
    assert ntiles <= 2048
    words = 2 * ntiles * 513 + 513
    assert lib.smr_align_workspace_size(ctypes.byref(a)) == 256 + ((words * 4 + 255) // 256) * 256


def test_route_align_workspace_follows_the_fused_align_cut_over(lib):
    """Behind a tcgen05 route, up to 704 slots are aligned by the route's last
    CTA in shared memory (no align scratch); above, the route counts its
    64-row tiles and the scan and scatter keep [tiles][E_al] counts and starts
    and [E_al] totals in the workspace."""
    def need(M):
        r = _good_route(M=M, H=1024, E=512, k=10, S=1)
        a = _set(_good_align(T=M, W=11, E_al=513, A=128), topk_ids=r.topk_ids)
        return lib.smr_route_align_workspace_size(ctypes.byref(r), ctypes.byref(a))
    assert need(64) == 256                      # 704 slots: fused
    tiles = -(-65 // 64)                        # 715 slots: counted, 2 tiles
    words = 2 * tiles * 513 + 513
    assert need(65) == 256 + ((words * 4 + 255) // 256) * 256
    tiles = -(-16384 // 64)
    words = 2 * tiles * 513 + 513
    assert need(16384) == 256 + ((words * 4 + 255) // 256) * 256


def test_route_align_consistency_checks(lib):
    r = _good_route()
    a = _good_align()
    a.topk_ids = r.topk_ids
    a.width = 10  # should be topk + S = 11
    assert lib.smr_route_align(ctypes.byref(r), ctypes.byref(a), None, 0, None) == _lib.SMR_ERR_INVALID_ARG
    assert "align.width must equal" in lib.smr_last_error().decode()


def test_tier_and_capacity_match_oracle(lib):
    for T, k, E in [(6, 8, 128), (1024, 8, 128), (2048, 8, 128), (4, 10, 512), (16384, 10, 512),
                    (0, 8, 128), (1, 1, 1)]:
        assert lib.smr_select_block_size(T, k, E) == oracle.select_block_size(T, k, E)
    for numel, E, A in [(1024, 128, 128), (1024, 128, 64), (8192, 128, 64), (44, 513, 64), (0, 1, 1)]:
        assert lib.smr_align_capacity(numel, E, A) == oracle.align_capacity(numel, E, A)
    assert lib.smr_select_block_size(5, 0, 8) == -1
    assert lib.smr_align_capacity(5, 0, 8) == -1


def test_disable_switch(monkeypatch):
    import moe_router_top_gb300 as smr
    monkeypatch.setenv("SMR_DISABLE", "1")
    with pytest.raises(smr.SmrUnsupported):
        smr.route(None, None, topk=1)


def test_route_profile_summary_parses():
    """The committed ncu summary of the route kernel carries the source hash
    and DRAM bytes per launch that bench.py reports as roofline traffic."""
    import hashlib
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "profiles", "tc_route_kernel_large_batch.md")).read()
    sha = re.search(r"- smr_tc\.cu sha256\[:16\]: `([0-9a-f]{16})`", text)
    dram = re.search(r"- dram bytes per launch: (\d+)", text)
    assert sha and dram
    import bench
    src = os.path.join(root, "moe_router_top_gb300", "csrc", "smr_tc.cu")
    current = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    expect = int(dram.group(1)) if sha.group(1) == current else None
    assert bench.traffic_from_profile() == expect


def _set(obj, **kw):
    for k, v in kw.items():
        setattr(obj, k, v)
    return obj


@pytest.mark.parametrize("change,status,fragment", [
    (dict(M=-1), _lib.SMR_ERR_INVALID_ARG, "M must be >= 0"),
    (dict(H=16392), _lib.SMR_ERR_INVALID_ARG, "H must be a multiple of 8 in [8, 16384]"),
    (dict(E=1025), _lib.SMR_ERR_INVALID_ARG, "E must be in [1, 1024]"),
    (dict(has_shared=2), _lib.SMR_ERR_INVALID_ARG, "has_shared must be 0 or 1"),
    (dict(topk=0), _lib.SMR_ERR_INVALID_ARG, "topk must be in [1, E]"),
    (dict(shared_scale=float("inf")), _lib.SMR_ERR_INVALID_ARG, "shared_scale must be finite"),
    (dict(ld_hidden=4100), _lib.SMR_ERR_INVALID_ARG, "ld_hidden must be >= H and a multiple of 8"),
    (dict(gate_w=0x20008), _lib.SMR_ERR_INVALID_ARG, "gate_w must be 16-byte aligned"),
    (dict(has_shared=0, topk=10), _lib.SMR_ERR_INVALID_ARG, "shared_w must be NULL when has_shared == 0"),
    (dict(bias=0x60002), _lib.SMR_ERR_INVALID_ARG, "bias must be 4-byte aligned"),
    (dict(topk_weights=0x50002), _lib.SMR_ERR_INVALID_ARG, "topk_weights must be 4-byte aligned"),
    (dict(logits_out=0x70008), _lib.SMR_ERR_INVALID_ARG, "logits_out must be 16-byte aligned"),
    (dict(renormalize=5), _lib.SMR_ERR_INVALID_ARG, "renormalize must be 0 or 1"),
    (dict(hidden_fp8=0x80000), _lib.SMR_ERR_INVALID_ARG, "hidden_scales is NULL"),
    (dict(hidden_fp8=0x80008, hidden_scales=0x90000), _lib.SMR_ERR_INVALID_ARG,
     "hidden_fp8 must be 16-byte aligned"),
    (dict(H=4104, ld_hidden=4104, hidden_fp8=0x80000, hidden_scales=0x90000),
     _lib.SMR_ERR_INVALID_ARG, "hidden_fp8 needs H % 128 == 0"),
])
def test_route_refuses_each_bad_argument(lib, change, status, fragment):
    """Every malformed route argument is refused before any launch, with its
    own reason in smr_last_error()."""
    a = _set(_good_route(), **change)
    assert lib.smr_route(ctypes.byref(a), None, 0, None) == status
    assert fragment in lib.smr_last_error().decode()
    assert lib.smr_last_launch_count() == 0


@pytest.mark.parametrize("change,status,fragment", [
    (dict(num_tokens=-1), _lib.SMR_ERR_INVALID_ARG, "num_tokens must be >= 0"),
    (dict(width=0), _lib.SMR_ERR_INVALID_ARG, "width must be >= 1"),
    (dict(num_experts=1026), _lib.SMR_ERR_INVALID_ARG, "num_experts must be in [1, 1025]"),
    (dict(block_size=4097), _lib.SMR_ERR_INVALID_ARG, "block_size must be 0 (M-aware tier) or in [1, 4096]"),
    (dict(topk_ids=0x10002), _lib.SMR_ERR_INVALID_ARG, "topk_ids must be 4-byte aligned"),
    (dict(sorted_token_ids=None), _lib.SMR_ERR_INVALID_ARG, "sorted_token_ids is NULL"),
    (dict(expert_ids=None), _lib.SMR_ERR_INVALID_ARG, "expert_ids is NULL"),
    (dict(expert_cap=3), _lib.SMR_ERR_INVALID_ARG, "expert_cap 3 < required"),
    (dict(num_tokens=1 << 25, width=64, sorted_cap=1 << 32, expert_cap=1 << 32),
     _lib.SMR_ERR_UNSUPPORTED, "num_tokens * width must be <= 2^30"),
])
def test_align_refuses_each_bad_argument(lib, change, status, fragment):
    a = _set(_good_align(), **change)
    assert lib.smr_align(ctypes.byref(a), None, 0, None) == status
    assert fragment in lib.smr_last_error().decode()
    assert lib.smr_last_launch_count() == 0


def test_static_entry_refuses_before_device_work(lib):
    """The no-allocation entry point checks its contract on the host, before
    it looks up its device array: M outside [1, 16] and scratch above the
    fixed array are refused."""
    r = _good_route(M=17, E=64)
    a = _set(_good_align(T=17, W=11, E_al=65), topk_ids=r.topk_ids)
    assert lib.smr_route_align_static(ctypes.byref(r), ctypes.byref(a), None) == _lib.SMR_ERR_UNSUPPORTED
    assert "1 <= M <= 16" in lib.smr_last_error().decode()
    r = _good_route(M=16, E=1024, k=10)  # 16 x 1024 tagged keys = 128 KiB: fits
    a = _set(_good_align(T=16, W=11, E_al=1025), topk_ids=r.topk_ids, width=11)
    need = lib.smr_route_align_workspace_size(ctypes.byref(r), ctypes.byref(a))
    assert need <= 256 * 1024


def test_failure_hook_and_static_error_refusals(lib):
    """The failure-injection hook takes only its sites and a positive limit;
    switching it off always succeeds. The fixed array's error getter refuses
    a NULL output before touching any device."""
    assert lib.smr_test_force_wait_timeout(7, 1) == _lib.SMR_ERR_INVALID_ARG
    assert "site must be" in lib.smr_last_error().decode()
    assert lib.smr_test_force_wait_timeout(_lib.SMR_STALL_TC_MERGE, 0) == _lib.SMR_ERR_INVALID_ARG
    assert lib.smr_test_force_wait_timeout(_lib.SMR_STALL_NONE, 0) == _lib.SMR_OK
    assert lib.smr_get_static_device_error(None, None) == _lib.SMR_ERR_INVALID_ARG


def test_align_eplb_arguments_checked(lib):
    """The EPLB remap's table pointers and sizes are checked before any
    launch, and the capacity is taken over the physical experts."""
    a = AlignArgs()
    a.topk_ids = 0x1000
    a.num_tokens, a.width, a.num_experts, a.block_size = 8, 4, 17, 16
    a.sorted_token_ids, a.expert_ids, a.num_tokens_post_padded = 0x2000, 0x3000, 0x4000
    a.eplb_map = 0x5002            # misaligned
    a.eplb_count = None
    a.eplb_max_replicas = 65       # above 64
    a.num_physical = 2000          # above 1025
    a.sorted_cap = a.expert_cap = 1 << 20
    assert lib.smr_align(ctypes.byref(a), None, 0, None) == _lib.SMR_ERR_INVALID_ARG
    msg = lib.smr_last_error().decode()
    for frag in ("eplb_count is NULL", "4-byte aligned", "eplb_max_replicas", "num_physical"):
        assert frag in msg, msg
    a.eplb_map, a.eplb_count, a.eplb_max_replicas, a.num_physical = 0x5000, 0x6000, 2, 40
    a.sorted_cap = 32 + 40 * 15 - 1  # one short of numel + num_physical * (A - 1)
    assert lib.smr_align(ctypes.byref(a), None, 0, None) == _lib.SMR_ERR_INVALID_ARG
    assert "required 632" in lib.smr_last_error().decode()
