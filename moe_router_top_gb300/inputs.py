"""Seeded synthetic inputs for the routing front-end (host side, numpy).

This module only draws and packages inputs. It holds none of the routing
arithmetic, so both the CUDA path and the CPU oracle can be fed from it
without sharing any method code.

bf16 tensors are returned as ``uint16`` arrays holding the bf16 bit
patterns. Normal draws are made in fp32 and rounded to bf16 (round to nearest
even) by PyTorch's dtype conversion, a library routine used by neither side.

Workloads (all synthetic; the pages' real activations and captured prefill
routing are not available):

* ``small_verify``   M=4, H=4096, E=512 + 1 shared, top-10, A=64
* ``tie_stress``     M in {1,3,8}, same shapes, every entry an integer in [-2, 2]
* ``short_prefill``  M=128, H=2048, E=128, top-8, no shared expert
* ``zipf_sweep``     M in {6,128,512,1024,2048}, as short_prefill plus a
  Zipf(s=1.1) log-prior bias over experts
* ``large_batch``    M=16384, H=4096, E=512 + 1 shared, top-10, A=128
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

SEED_BASE = 20261202


def seed_for(config_index: int, variant: int = 0) -> int:
    """Seed recipe: 20261202 + 100 * config index + variant."""
    return SEED_BASE + 100 * int(config_index) + int(variant)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (RNE) with torch's dtype conversion."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class RouteInputs:
    M: int
    H: int
    E: int
    topk: int
    has_shared: int
    shared_scale: float
    x: np.ndarray                    # uint16 [M, H] bf16 bits
    w: np.ndarray                    # uint16 [E, H] bf16 bits
    ws: Optional[np.ndarray]         # uint16 [1, H] bf16 bits, or None
    bias: Optional[np.ndarray]       # float32 [E], or None
    block_size: int = 0              # 0 = M-aware tier
    name: str = ""
    renormalize: bool = True         # routing variant flags (passed through, no arithmetic here)
    shared_bf16: bool = False

    @property
    def width(self) -> int:
        return self.topk + self.has_shared

    @property
    def num_experts_align(self) -> int:
        return self.E + self.has_shared


def _normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def _int_bf16(rng: np.random.Generator, shape, lo: int = -2, hi: int = 2) -> np.ndarray:
    return f32_to_bf16_bits(rng.integers(lo, hi + 1, size=shape).astype(np.float32))


def zipf_log_prior(E: int, s: float, rng: np.random.Generator) -> np.ndarray:
    """Bias b[e] = -s * ln(rank_e), rank a seeded permutation of 1..E (fp32).

    Adding it to the logits multiplies the softmax prior of expert e by
    rank_e ** -s, a Zipf(s) law over experts (the normaliser cancels).
    """
    ranks = rng.permutation(E).astype(np.float64) + 1.0
    return (-s * np.log(ranks)).astype(np.float32)


def make_route_inputs(M: int, H: int, E: int, topk: int, has_shared: int, *,
                      seed: int, dist: str = "normal", x_std: float = 1.0,
                      w_std: float = 0.02, zipf_s: Optional[float] = None,
                      shared_scale: float = 1.0, block_size: int = 0,
                      name: str = "", renormalize: bool = True,
                      shared_bf16: bool = False) -> RouteInputs:
    rng = np.random.default_rng(seed)
    if dist == "normal":
        x = _normal_bf16(rng, (M, H), x_std)
        w = _normal_bf16(rng, (E, H), w_std)
        ws = _normal_bf16(rng, (1, H), w_std) if has_shared else None
    elif dist == "int":
        x = _int_bf16(rng, (M, H))
        w = _int_bf16(rng, (E, H))
        ws = _int_bf16(rng, (1, H)) if has_shared else None
    else:
        raise ValueError(f"unknown dist {dist!r}")
    bias = zipf_log_prior(E, zipf_s, rng) if zipf_s is not None else None
    return RouteInputs(M=M, H=H, E=E, topk=topk, has_shared=has_shared,
                       shared_scale=float(shared_scale), x=x, w=w, ws=ws,
                       bias=bias, block_size=block_size, name=name,
                       renormalize=renormalize, shared_bf16=shared_bf16)


# --- the five workloads -----------------------------------------------------

def small_verify(M: int = 4, variant: int = 0) -> RouteInputs:
    return make_route_inputs(M, 4096, 512, 10, 1, seed=seed_for(0, variant),
                             block_size=64, name=f"small_verify_M{M}")


def tie_stress(M: int, variant: int = 0) -> RouteInputs:
    return make_route_inputs(M, 4096, 512, 10, 1, seed=seed_for(1, variant + M),
                             dist="int", block_size=64, name=f"tie_stress_M{M}")


def short_prefill(block_size: int = 0, variant: int = 0) -> RouteInputs:
    return make_route_inputs(128, 2048, 128, 8, 0, seed=seed_for(2, variant),
                             block_size=block_size, name=f"short_prefill_A{block_size}")


ZIPF_TOKENS = (6, 128, 512, 1024, 2048)


def zipf_sweep(M: int, variant: int = 0) -> RouteInputs:
    return make_route_inputs(M, 2048, 128, 8, 0, seed=seed_for(3, variant + M),
                             zipf_s=1.1, block_size=0, name=f"zipf_M{M}")


def large_batch(M: int = 16384, variant: int = 0) -> RouteInputs:
    return make_route_inputs(M, 4096, 512, 10, 1, seed=seed_for(4, variant),
                             block_size=128, name=f"large_batch_M{M}")


def random_ids(num_tokens: int, width: int, num_experts: int, *, seed: int,
               unique_rows: bool = True, skew: Optional[float] = None) -> np.ndarray:
    """Random expert ids [num_tokens, width] int32 for align-only tests.

    unique_rows draws each row without replacement (as top-k does); skew, if
    given, draws experts with Zipf(skew) weights so a few experts are hot.
    """
    rng = np.random.default_rng(seed)
    out = np.empty((num_tokens, width), dtype=np.int32)
    p = None
    if skew is not None:
        p = (np.arange(1, num_experts + 1, dtype=np.float64) ** -skew)
        p = p[rng.permutation(num_experts)]
        p /= p.sum()
    for t in range(num_tokens):
        if unique_rows:
            out[t] = rng.choice(num_experts, size=width, replace=False, p=p)
        else:
            out[t] = rng.choice(num_experts, size=width, replace=True, p=p)
    return out


def random_eplb_map(num_experts: int, max_replicas: int, num_physical: int, *,
                    seed: int):
    """A random expert-parallel load-balancing table: each logical expert
    gets 1..max_replicas replicas (int32 count [num_experts]), each replica a
    distinct physical expert (int32 map [num_experts, max_replicas], unused
    entries -1); needs num_physical >= the replicas drawn (checked)."""
    rng = np.random.default_rng(seed)
    count = rng.integers(1, max_replicas + 1, size=num_experts).astype(np.int32)
    while int(count.sum()) > num_physical:
        count[int(np.argmax(count))] -= 1
    phys = rng.permutation(num_physical)[: int(count.sum())].astype(np.int32)
    emap = np.full((num_experts, max_replicas), -1, np.int32)
    pos = 0
    for e in range(num_experts):
        emap[e, : count[e]] = phys[pos: pos + count[e]]
        pos += int(count[e])
    return emap, count
