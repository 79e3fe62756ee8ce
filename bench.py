#!/usr/bin/env python3
"""Benchmark of the routing front-end on one GB300 (or N replicas).

One step = route + align of one batch through the C ABI (libsmr.so):
the headline workload is the large batch, M=16384 tokens, H=4096, E=512
routed experts + 1 shared, top-10 renormalised + shared slot, align at A=128.
Printed as ONE JSON line by rank 0:

  value        routed tokens/s, inputs resident in HBM (two alternating
               [16384, 4096] bf16 hidden-state buffers, 134 MB each, larger
               than the 126.5 MiB L2; the 4.2 MB gate stays resident)
  e2e          same metric with the hidden states copied host->device
               (pinned) and all outputs copied back inside the timed region
  roofline     the tcgen05 route kernel against the measured bf16 tensor peak
  small_m      us per route+align call at M=4 and M=8 (one launch each),
               CUDA graph of back-to-back calls over a ring of gate/hidden
               copies larger than L2, against the measured HBM peak
  cpu_baseline the C oracle on a bounded sample of the same workload

`--impl reference` times the oracle itself (the slow CPU definition) on a
bounded sample per step and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("µs per route+align call at M=4/8 and routed tokens/s at M=16K; "
          "% of roofline")
M_LARGE, H, E, K, S, A_LARGE = 16384, 4096, 512, 10, 1, 128
GRAPH_STEPS = 50               # route_align steps per captured CUDA graph (at most)
WORKLOAD = ("large_batch: M=16384 tokens, H=4096, E=512 routed + 1 shared gate, "
            "top-10 softmax+renormalize + shared slot, route + align at A=128")
ORACLE_SAMPLE_ROWS = 1024      # cpu_baseline, single-threaded leg: rows of the large batch
REFERENCE_BUDGET_S = 90.0      # --impl reference: whole run, warm-up included


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """Polls SM clock and clocks-event reasons through NVML (read-only)."""

    REASONS = {0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x1: "gpu_idle", 0x10: "sync_boost", 0x100: "display_clock_setting"}

    def __init__(self, index: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        if vis and all(v.strip().isdigit() for v in vis.split(",")):
            index = int(vis.split(",")[index])
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        self._stop = threading.Event()
        self._nvml = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) != 0:
                return
            self._nvml, self._h = nv, h
            self._reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
        except OSError:
            pass

    def _run(self):
        nv, h = self._nvml, self._h
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if self._reasons_fn(h, ctypes.byref(rs)) == 0:
                self.reasons |= rs.value
            time.sleep(0.0002)

    def __enter__(self):
        if self._nvml is not None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        if self._nvml is not None:
            self._stop.set()
            self._t.join()

    def summary(self):
        reasons = [n for bit, n in self.REASONS.items() if self.reasons & bit and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(self.samples)}


# --------------------------------------------------------------- helpers ----

def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "smr" else "gloo"
        if args.impl == "smr":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif args.impl == "smr":
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Whole-job tokens/s of `world` replicas, each routing its own batch of
    tokens_per_rank tokens per step; ms_per_step is the slowest rank's step
    time (max over ranks), so the job's rate is set by that rank."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


def to_dev_bf16(a, torch):
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def traffic_from_profile():
    """dram bytes per launch of the route kernel from the committed ncu
    summary, or None if the kernel source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "tc_route_kernel_large_batch.md")
    src = os.path.join(ROOT, "moe_router_top_gb300", "csrc", "smr_tc.cu")
    try:
        text = open(path).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ": " in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(": ", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("smr_tc.cu sha256[:16]") != sha:
        return None
    try:
        return int(vals["dram bytes per launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------- smr arm ------

def bench_large(args, world, rank, torch, smr, inputs):
    import numpy as np
    ri = inputs.large_batch(variant=rank)
    xs = [to_dev_bf16(ri.x, torch)]
    x2 = torch.empty_like(xs[0])
    x2.copy_(xs[0].roll(1, dims=0))
    xs.append(x2)
    w = to_dev_bf16(ri.w, torch)
    ws = to_dev_bf16(ri.ws, torch)
    M = ri.M
    width = K + S
    ids = torch.empty((M, width), dtype=torch.int32, device="cuda")
    wts = torch.empty((M, width), dtype=torch.float32, device="cuda")
    cap = smr.align_capacity(M * width, E + S, A_LARGE)
    srt = torch.empty(cap, dtype=torch.int32, device="cuda")
    eids = torch.empty((cap + A_LARGE - 1) // A_LARGE, dtype=torch.int32, device="cuda")
    npp = torch.empty(1, dtype=torch.int32, device="cuda")
    wsp = smr.Workspace()
    stream = torch.cuda.current_stream()

    def step(i):
        # one call of the public route+align entry point (the route kernel also
        # counts the experts of its rows for the align launches behind it)
        smr.route_align(xs[i & 1], w, ws, topk=K, block_size=A_LARGE, topk_ids=ids,
                        topk_weights=wts, sorted_token_ids=srt, expert_ids=eids,
                        num_tokens_post_padded=npp, workspace=wsp)

    for i in range(args.warmup):
        step(i)
    launches_per_step = smr.last_launch_count()
    torch.cuda.synchronize()

    # the timed steps run as replays of a CUDA graph of G steps (as a serving
    # loop would), plus any remainder eagerly: exactly args.steps steps
    G = min(args.steps, GRAPH_STEPS)
    cap_stream = torch.cuda.Stream()
    cap_stream.wait_stream(stream)
    with torch.cuda.stream(cap_stream):
        for i in range(3):
            step(i)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap_stream):
        for i in range(G):
            step(i)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    replays, rest = divmod(args.steps, G)

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device())
    barrier(world)
    torch.cuda.synchronize()
    with sampler:
        start.record(stream)
        for _ in range(replays):
            graph.replay()
        for i in range(rest):
            step(i)
        end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = start.elapsed_time(end) / args.steps
    assert smr.get_device_error(wsp) == 0

    # the route kernel alone (roofline): route-only calls on the same
    # alternating inputs, replayed from a CUDA graph of RG launches (so host
    # submission never shows in the interval), CUDA events on the replay
    # stream around each replay; per launch = replay time / RG
    RG = 20
    with torch.cuda.stream(cap_stream):
        for i in range(3):
            smr.route(xs[i & 1], w, ws, topk=K, topk_ids=ids, topk_weights=wts, workspace=wsp)
    torch.cuda.synchronize()
    rgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(rgraph, stream=cap_stream):
        for i in range(RG):
            smr.route(xs[i & 1], w, ws, topk=K, topk_ids=ids, topk_weights=wts, workspace=wsp)
    rgraph.replay()
    torch.cuda.synchronize()
    n_rep = max(3, min(args.steps // RG, 25))
    route_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(n_rep)]
    for a, b in route_ev:
        a.record(stream)
        rgraph.replay()
        b.record(stream)
    torch.cuda.synchronize()
    route_ms = statistics.median(a.elapsed_time(b) for a, b in route_ev) / RG
    assert smr.get_device_error(wsp) == 0

    # e2e: hidden states from pinned host memory, outputs back to the host
    hx = torch.from_numpy(np.ascontiguousarray(ri.x).view(np.int16)).view(torch.bfloat16).pin_memory()
    h_ids = torch.empty_like(ids, device="cpu").pin_memory()
    h_wts = torch.empty_like(wts, device="cpu").pin_memory()
    h_srt = torch.empty_like(srt, device="cpu").pin_memory()
    h_eids = torch.empty_like(eids, device="cpu").pin_memory()
    h_npp = torch.empty_like(npp, device="cpu").pin_memory()
    h2d = hx.numel() * 2
    d2h = (ids.numel() + wts.numel() + srt.numel() + eids.numel() + npp.numel()) * 4

    def e2e_step():
        xs[0].copy_(hx, non_blocking=True)
        step(0)
        h_ids.copy_(ids, non_blocking=True)
        h_wts.copy_(wts, non_blocking=True)
        h_srt.copy_(srt, non_blocking=True)
        h_eids.copy_(eids, non_blocking=True)
        h_npp.copy_(npp, non_blocking=True)

    n_e2e = max(3, min(args.steps, 50))
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    e2.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = s2.elapsed_time(e2) / n_e2e

    # e2e as a serving loop runs it: step i+1's hidden states cross the host
    # link (copy stream) while step i routes (compute stream); two device
    # buffers, events order every reuse. Every step's host->device copy and
    # its outputs' device->host copy are inside the timed region.
    copy_s = torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    for ev in consumed:
        ev.record(stream)

    def e2e_pipelined(n):
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(copy_s):
                copy_s.wait_event(consumed[b])  # step i-2 is done with buffer b
                xs[b].copy_(hx, non_blocking=True)
                copied[b].record(copy_s)
            stream.wait_event(copied[b])
            step(b)
            consumed[b].record(stream)
            h_ids.copy_(ids, non_blocking=True)
            h_wts.copy_(wts, non_blocking=True)
            h_srt.copy_(srt, non_blocking=True)
            h_eids.copy_(eids, non_blocking=True)
            h_npp.copy_(npp, non_blocking=True)

    e2e_pipelined(3)
    torch.cuda.synchronize()
    barrier(world)
    s3, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s3.record(stream)
    e2e_pipelined(n_e2e)
    stream.wait_stream(copy_s)
    e3.record(stream)
    torch.cuda.synchronize()
    e2e_ms = s3.elapsed_time(e3) / n_e2e
    return {"ms": ms, "route_ms": route_ms, "e2e_ms": e2e_ms, "e2e_serial_ms": e2e_serial_ms,
            "h2d": h2d, "d2h": d2h, "graph_steps": G, "replays": replays, "eager_steps": rest,
            "launches_per_step": launches_per_step, "clocks": sampler.summary(), "ri": ri,
            "ids": ids, "M": M}


def bench_small(torch, smr, inputs, M, l2_bytes, reps=20, calls=100):
    """us per route+align call at small M, weights streamed from HBM."""
    ri = inputs.small_verify(M)
    gate_bytes = (E + S) * H * 2
    ncopies = max(2, int(2 * l2_bytes // gate_bytes) + 1)
    ws_list = [to_dev_bf16(ri.w, torch) for _ in range(ncopies)]
    wsh = [to_dev_bf16(ri.ws, torch) for _ in range(ncopies)]
    x_list = [to_dev_bf16(ri.x, torch) for _ in range(ncopies)]
    width = K + S
    ids = torch.empty((M, width), dtype=torch.int32, device="cuda")
    wts = torch.empty((M, width), dtype=torch.float32, device="cuda")
    A = 64
    cap = smr.align_capacity(M * width, E + S, A)
    srt = torch.empty(cap, dtype=torch.int32, device="cuda")
    eids = torch.empty((cap + A - 1) // A, dtype=torch.int32, device="cuda")
    npp = torch.empty(1, dtype=torch.int32, device="cuda")
    wsp = smr.Workspace()

    def call(j):
        smr.route_align(x_list[j], ws_list[j], wsh[j], topk=K, block_size=A, topk_ids=ids,
                        topk_weights=wts, sorted_token_ids=srt, expert_ids=eids,
                        num_tokens_post_padded=npp, workspace=wsp)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for j in range(3):
            call(j)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    launches = smr.last_launch_count()

    def graph_time(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for c in range(calls):
                call(c % copies)
        g.replay()
        torch.cuda.synchronize()
        times = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b) * 1000.0 / calls)
        return statistics.median(times)

    us_hbm = graph_time(ncopies)
    us_hot = graph_time(1)
    # eager: one call per event pair
    eager = []
    for j in range(50):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call(j % ncopies)
        b.record()
        torch.cuda.synchronize()
        eager.append(a.elapsed_time(b) * 1000.0)
    bytes_moved = gate_bytes + M * H * 2 + M * width * 8
    return {"us_per_call": us_hbm, "us_hot_l2": us_hot, "us_eager": statistics.median(eager),
            "bytes": bytes_moved, "launches": launches, "ring_copies": ncopies}


def bench_consumer(torch, smr, inputs, N=1536, reps=10, calls=20):
    """The M-aware tier end to end: route_align + the consumer expert GEMM
    (bf16 experts [128, N, 2048], N = 1536 for a gate+up projection of 768)
    on the skewed sweep's batches, at A = 64 and A = 128. The expert GEMM's
    work follows npp (blocks at or past it return at once)."""
    H_, E_, K_ = 2048, 128, 8
    g = torch.Generator(device="cuda").manual_seed(7)
    ew = (torch.randn((E_, N, H_), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    out_all = {}
    for M in inputs.ZIPF_TOKENS[1:]:
        ri = inputs.zipf_sweep(M)
        x = to_dev_bf16(ri.x, torch)
        w = to_dev_bf16(ri.w, torch)
        b = torch.from_numpy(ri.bias).cuda()
        row = {"tier_block_size": smr.select_block_size(M, K_, E_), "routed_rows": M * K_}
        for A in (64, 128):
            wsp = smr.Workspace()
            ids, wts, srt, eids, npp = smr.route_align(x, w, None, b, topk=K_, block_size=A, workspace=wsp)
            out = torch.empty((M * K_, N), dtype=torch.float32, device="cuda")

            def step(gemm_only=False):
                if not gemm_only:
                    smr.route_align(x, w, None, b, topk=K_, block_size=A, topk_ids=ids, topk_weights=wts,
                                    sorted_token_ids=srt, expert_ids=eids, num_tokens_post_padded=npp,
                                    workspace=wsp)
                smr.expert_gemm(x, ew, srt, eids, npp, width=K_, block_size=A, out=out, workspace=wsp)

            def time_graph(gemm_only):
                st = torch.cuda.Stream()
                st.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(st):
                    step(gemm_only)
                torch.cuda.current_stream().wait_stream(st)
                torch.cuda.synchronize()
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr):
                    for _ in range(calls):
                        step(gemm_only)
                gr.replay()
                torch.cuda.synchronize()
                ts = []
                for _ in range(reps):
                    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    gr.replay()
                    e.record()
                    torch.cuda.synchronize()
                    ts.append(a.elapsed_time(e) * 1000.0 / calls)
                return statistics.median(ts)

            us_gemm = time_graph(True)
            us_step = time_graph(False)
            n = int(npp.item())
            row[f"A{A}"] = {"npp": n, "padding_fraction": 1.0 - M * K_ / n,
                            "us_route_align_plus_expert_gemm": us_step, "us_expert_gemm": us_gemm,
                            "expert_gemm_useful_tflops": 2.0 * M * K_ * N * H_ / (us_gemm * 1e-6) / 1e12,
                            "expert_gemm_done_tflops": 2.0 * n * N * H_ / (us_gemm * 1e-6) / 1e12}
            assert smr.get_device_error(wsp) == 0
        out_all[f"M{M}"] = row
    return {"workload": f"skewed sweep (H=2048, E=128, top-8, Zipf 1.1 bias), expert GEMM N={N} bf16",
            "timing": f"CUDA graph of {calls} steps, median of {reps} replays", "by_tokens": out_all}


def cpu_baseline_large():
    """The C oracle on the large batch: all 16384 rows split over every host
    core (median of 3 runs), and single-threaded on the first
    ORACLE_SAMPLE_ROWS rows."""
    import numpy as np
    import oracle
    from moe_router_top_gb300 import inputs
    ri = inputs.large_batch()
    cores = host_cores()

    def run(rows, threads):
        t0 = time.perf_counter()
        r = oracle.route(ri.x, ri.w, ri.ws, None, K, 1.0, rows=rows, threads=threads)
        oracle.align(r.ids, E + S, A_LARGE)
        return time.perf_counter() - t0

    all_rows = np.arange(ri.M)
    mt = sorted(run(all_rows, cores) for _ in range(3))
    st = run(np.arange(ORACLE_SAMPLE_ROWS), 1)
    return {"value": ri.M / mt[1], "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"all {ri.M} rows of the large batch, route + align, C oracle with the rows "
                      f"split over {cores} host threads; median of 3 runs "
                      f"({', '.join(f'{t:.2f}' for t in mt)} s)",
            "single_thread": {"value": ORACLE_SAMPLE_ROWS / st, "unit": "tokens/s", "cores": 1,
                              "sample": f"first {ORACLE_SAMPLE_ROWS} rows, one thread ({st:.2f} s)"}}


def cpu_baseline_small(M):
    """The C oracle's route + align of one small_verify call (median of 3)."""
    import oracle
    from moe_router_top_gb300 import inputs
    ri = inputs.small_verify(M)
    times = []
    for _ in range(3):
        t0 = time.perf_counter()
        r = oracle.route(ri.x, ri.w, ri.ws, None, K, 1.0)
        oracle.align(r.ids, E + S, 64)
        times.append(time.perf_counter() - t0)
    times.sort()
    return {"value": times[1] * 1e6, "unit": "us per call", "cores": 1, "kind": "oracle",
            "sample": f"one M={M} route + align call (the whole workload), single-threaded C oracle, "
                      f"median of 3"}


def run_smr(args):
    import torch
    world, rank, local = dist_setup(args)
    import moe_router_top_gb300 as smr
    from moe_router_top_gb300 import build, inputs
    build.build()
    hbm_gbs, tc_tflops, src = peaks()
    if args.no_large:
        line = {"metric": METRIC, "partial": "small-batch timings only"}
        l2 = torch.cuda.get_device_properties(0).L2_cache_size
        line["small_m"] = {f"M{M}": bench_small(torch, smr, inputs, M, l2) for M in (4, 8)}
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    res = bench_large(args, world, rank, torch, smr, inputs)
    ms = max_over_ranks(world, res["ms"])
    e2e_ms = max_over_ranks(world, res["e2e_ms"])
    e2e_serial_ms = max_over_ranks(world, res["e2e_serial_ms"])
    flops = 2.0 * M_LARGE * H * (E + S)
    achieved = flops / (res["route_ms"] * 1e-3) / 1e12
    line = {
        "metric": METRIC,
        "value": replica_throughput(world, M_LARGE, ms),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) hidden states, N(0,0.02) gate weights)",
        "config": {"workload": WORKLOAD, "M": M_LARGE, "H": H, "E": E, "shared": S, "topk": K,
                   "block_size": A_LARGE, "parallelism": f"replicas{world}",
                   "l2": "inputs larger than L2: two alternating 134 MB hidden-state buffers",
                   "timing": (f"route_align steps: {res['replays']} replay(s) of a CUDA graph of "
                              f"{res['graph_steps']} steps" +
                              (f" + {res['eager_steps']} eager steps" if res["eager_steps"] else ""))},
        "e2e": {"value": replica_throughput(world, M_LARGE, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "timing": "route_align through the public API; each step's hidden states copied "
                          "from pinned host memory and all its outputs copied back, inside the "
                          "timed region; the next step's copy overlaps this step's routing "
                          "(two device buffers, a copy stream)",
                "serial_value": replica_throughput(world, M_LARGE, e2e_serial_ms)},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tc_tflops,
                     "unit": "TFLOP/s", "frac": achieved / tc_tflops,
                     "traffic": traffic_from_profile(),
                     "kernel": "tc_route_kernel (gate GEMM + fused top-k epilogue)",
                     "kernel_us": res["route_ms"] * 1000.0,
                     "kernel_timing": "route-only launches on the same alternating inputs, replayed "
                                      "from a CUDA graph of 20; CUDA events on the stream around "
                                      "each replay (median) / 20, inter-launch gaps included",
                     "peak_source": f"{src} bf16 dense (burst)"},
        "gpu_launches": res["launches_per_step"] * args.steps,
        "clocks": res["clocks"],
    }
    if rank == 0 and not args.no_small:
        l2 = torch.cuda.get_device_properties(0).L2_cache_size
        small = {}
        for M in (4, 8):
            r = bench_small(torch, smr, inputs, M, l2)
            t_roof = r["bytes"] / (hbm_gbs * 1e9) * 1e6
            small[f"M{M}"] = {"us_per_call": r["us_per_call"], "us_hot_l2": r["us_hot_l2"],
                              "us_eager": r["us_eager"], "launches_per_call": r["launches"],
                              "roofline": {"bound": "hbm", "bytes": r["bytes"],
                                           "achieved_gbs": r["bytes"] / (r["us_per_call"] * 1e-6) / 1e9,
                                           "peak_gbs": hbm_gbs, "frac": t_roof / r["us_per_call"],
                                           "peak_source": src},
                              "timing": f"CUDA graph of 100 calls over {r['ring_copies']} gate/hidden "
                                        f"copies (> 2x L2), median of 20 replays; a call may launch "
                                        f"during the previous call's tail (programmatic dependent "
                                        f"launch) and stream its gate before waiting for it"}
            if not args.no_cpu:
                small[f"M{M}"]["cpu_baseline"] = cpu_baseline_small(M)
        line["small_m"] = small
    if rank == 0 and not args.no_consumer:
        line["consumer_tier"] = bench_consumer(torch, smr, inputs)
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline_large()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------- reference arm ------

def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import oracle
    from moe_router_top_gb300 import inputs
    oracle.build()
    ri = inputs.large_batch()
    cores = host_cores()
    t0 = time.perf_counter()
    oracle.route(ri.x, ri.w, ri.ws, None, K, 1.0, rows=np.arange(2 * cores), threads=cores)
    per_row = (time.perf_counter() - t0) / (2 * cores)
    rows_per_step = int(max(cores, min(64 * cores,
                                       REFERENCE_BUDGET_S / ((args.steps + args.warmup) * per_row))))

    def step(i):
        rows = (np.arange(rows_per_step) + i * rows_per_step) % ri.M
        r = oracle.route(ri.x, ri.w, ri.ws, None, K, 1.0, rows=rows, threads=cores)
        oracle.align(r.ids, E + S, A_LARGE)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = args.steps * rows_per_step / dt
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dt * 1000.0 / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) hidden states, N(0,0.02) gate weights)",
        "config": {"workload": WORKLOAD, "M": M_LARGE, "H": H, "E": E, "shared": S, "topk": K,
                   "block_size": A_LARGE, "parallelism": "host cores, rank 0 only"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows_per_step} rows of the large batch per step, "
                                   f"route + align, C oracle with the rows split over {cores} "
                                   f"host threads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_profile(args):
    """A few route+align steps at --profile-m tokens (large-batch shapes), for
    ncu captures of single launches on a small case."""
    import torch
    import moe_router_top_gb300 as smr
    from moe_router_top_gb300 import build, inputs
    build.build()
    torch.cuda.set_device(0)
    ri = inputs.large_batch(args.profile_m)
    x, w, ws = (to_dev_bf16(a, torch) for a in (ri.x, ri.w, ri.ws))
    wsp = smr.Workspace()
    for _ in range(args.warmup + args.steps):
        smr.route_align(x, w, ws, topk=K, block_size=A_LARGE, workspace=wsp)
    torch.cuda.synchronize()
    assert smr.get_device_error(wsp) == 0
    print(f"profile run: {args.steps} steps at M={args.profile_m}")


def run_profile_expert(args):
    """A few route_align + expert GEMM steps on the skewed sweep's shapes at
    --profile-expert tokens (A = 128, N = 1536), for ncu captures."""
    import torch
    import moe_router_top_gb300 as smr
    from moe_router_top_gb300 import build, inputs
    build.build()
    torch.cuda.set_device(0)
    ri = inputs.zipf_sweep(args.profile_expert)
    x, w = to_dev_bf16(ri.x, torch), to_dev_bf16(ri.w, torch)
    b = torch.from_numpy(ri.bias).cuda()
    g = torch.Generator(device="cuda").manual_seed(7)
    ew = (torch.randn((128, 1536, 2048), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    wsp = smr.Workspace()
    for _ in range(args.warmup + args.steps):
        ids, wts, srt, eids, npp = smr.route_align(x, w, None, b, topk=8, block_size=128, workspace=wsp)
        smr.expert_gemm(x, ew, srt, eids, npp, width=8, block_size=128, workspace=wsp)
    torch.cuda.synchronize()
    assert smr.get_device_error(wsp) == 0
    print(f"profile run: {args.steps} steps of route_align + expert GEMM at M={args.profile_expert}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("smr", "reference"), default="smr")
    ap.add_argument("--no-small", action="store_true", help="skip the M=4/8 small-batch timings")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-consumer", action="store_true",
                    help="skip the route_align + expert GEMM timings at both block sizes")
    ap.add_argument("--no-large", action="store_true",
                    help="only the M=4/8 small-batch timings (prints a partial line)")
    ap.add_argument("--profile-m", type=int, default=0,
                    help="profiling aid: run `--steps` route+align steps of the large-batch "
                         "shapes at this many tokens and exit (no JSON line)")
    ap.add_argument("--profile-expert", type=int, default=0,
                    help="profiling aid: route_align + expert GEMM steps on the skewed sweep's "
                         "shapes at this many tokens, then exit (no JSON line)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.profile_expert:
        run_profile_expert(args)
    elif args.profile_m:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_smr(args)


if __name__ == "__main__":
    main()
