"""Seeded synthetic inputs for the NVFP4-weight MoE layer.

This module draws random numbers and nothing else: it holds none of the
layer's arithmetic (no quantisation, routing, planning or GEMM), so that the
CPU oracle and the CUDA path can both take their inputs from it.

The pages measure the layer on a real checkpoint (512 experts, top-10, FP16
activations, NVFP4 weights) with synthetic activations ("[Kernel][SM70]
Improve Qwen3.8 no-MTP concurrency", section "Latest grouped-MoE screen").
That checkpoint is not available, so every tensor here is drawn from a seeded
PCG64 stream:

* x ~ N(0, 1) rounded to FP16, shape [M, H];
* router weight W_r ~ N(0, 0.02) rounded to FP16, shape [H, E];
* expert weights ~ N(0, 0.02) in FP32: W13 [2I, H] (gate rows then up rows)
  and W2 [H, I], drawn one expert at a time, to be quantised to NVFP4 by the
  caller;
* "bias" workloads: a per-expert FP32 router bias ~ N(0, 1);
* "zipf" workloads: bias_e = -1.2 * ln(rank_e), ranks 1..E assigned by a
  seeded permutation (the log of an unnormalised Zipf(1.2) probability), plus
  a shared expert and a gate vector w_g ~ N(0, 0.02) FP16 [H].

Seeds: tensor stream = SeedSequence([1000 * config_index + tensor_id, sub]).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# tensor ids used in seeds
_X, _WR, _BIAS, _W13, _W2, _S13, _S2, _WG, _PERM = 1, 2, 3, 4, 5, 6, 7, 8, 9


@dataclass(frozen=True)
class Workload:
    name: str
    index: int          # seed family
    M: int              # tokens
    H: int              # hidden size
    E: int              # routed experts
    k: int              # experts per token
    I: int              # expert intermediate size
    bias: str = "none"  # "none" | "normal" | "zipf"
    shared: bool = False

    @property
    def pairs(self) -> int:
        return self.M * self.k


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_m8", 0, 8, 256, 16, 2, 128),
        Workload("decode_m1", 1, 1, 2048, 512, 10, 512),
        Workload("decode_m16_bias", 2, 16, 2048, 512, 10, 512, bias="normal"),
        Workload("prefill_m8192", 3, 8192, 2048, 512, 10, 512),
        Workload("prefill_m8192_zipf_shared", 4, 8192, 2048, 512, 10, 512,
                 bias="zipf", shared=True),
        # the pages' M784 point (a prefill chunk; the grouped path's lower range)
        Workload("prefill_m784", 3, 784, 2048, 512, 10, 512),
    ]
}


def _rng(wl: Workload, tensor: int, sub: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(
        np.random.SeedSequence([1000 * wl.index + tensor, sub])))


def with_tokens(wl: Workload, M: int) -> Workload:
    """The same layer shapes and seeds with a different token count."""
    return Workload(wl.name, wl.index, M, wl.H, wl.E, wl.k, wl.I, wl.bias, wl.shared)


def custom(name: str, M: int, H: int, E: int, k: int, I: int, bias: str = "none",
           shared: bool = False, index: int = 90) -> Workload:
    return Workload(name, index, M, H, E, k, I, bias, shared)


def activations(wl: Workload, variant: int = 0) -> np.ndarray:
    """x: FP16 [M, H] ~ N(0, 1)."""
    r = _rng(wl, _X, variant)
    return r.standard_normal((wl.M, wl.H), dtype=np.float32).astype(np.float16)


def router_weight(wl: Workload) -> np.ndarray:
    """W_r: FP16 [H, E] ~ N(0, 0.02)."""
    r = _rng(wl, _WR)
    return (r.standard_normal((wl.H, wl.E), dtype=np.float32) * np.float32(0.02)).astype(np.float16)


def router_bias(wl: Workload):
    """FP32 [E] or None."""
    if wl.bias == "none":
        return None
    if wl.bias == "normal":
        return _rng(wl, _BIAS).standard_normal((wl.E,), dtype=np.float32)
    if wl.bias == "zipf":
        ranks = _rng(wl, _PERM).permutation(wl.E) + 1
        return (-1.2 * np.log(ranks.astype(np.float64))).astype(np.float32)
    raise ValueError(wl.bias)


def gate_weight(wl: Workload):
    """w_g: FP16 [H] ~ N(0, 0.02), or None without a shared expert."""
    if not wl.shared:
        return None
    r = _rng(wl, _WG)
    return (r.standard_normal((wl.H,), dtype=np.float32) * np.float32(0.02)).astype(np.float16)


def expert_w13(wl: Workload, e: int) -> np.ndarray:
    """FP32 [2I, H] ~ N(0, 0.02): rows 0..I-1 gate, rows I..2I-1 up."""
    r = _rng(wl, _W13, e)
    return r.standard_normal((2 * wl.I, wl.H), dtype=np.float32) * np.float32(0.02)


def expert_w2(wl: Workload, e: int) -> np.ndarray:
    """FP32 [H, I] ~ N(0, 0.02)."""
    r = _rng(wl, _W2, e)
    return r.standard_normal((wl.H, wl.I), dtype=np.float32) * np.float32(0.02)


def shared_w13(wl: Workload) -> np.ndarray:
    r = _rng(wl, _S13)
    return r.standard_normal((2 * wl.I, wl.H), dtype=np.float32) * np.float32(0.02)


def shared_w2(wl: Workload) -> np.ndarray:
    r = _rng(wl, _S2)
    return r.standard_normal((wl.H, wl.I), dtype=np.float32) * np.float32(0.02)


def all_w13(wl: Workload, experts=None) -> np.ndarray:
    ex = range(wl.E) if experts is None else experts
    return np.stack([expert_w13(wl, e) for e in ex])


def all_w2(wl: Workload, experts=None) -> np.ndarray:
    ex = range(wl.E) if experts is None else experts
    return np.stack([expert_w2(wl, e) for e in ex])


# ---- dense few-row projections ---------------------------------------------------
# The pages measure the QPN2 / QPN8 projections on a dense model's MLP split
# four ways (gate/up and down projections, M = 8 / 16 / 32) without giving
# the sizes; these stand-ins are hidden 5120 and intermediate 17408 split four
# ways: gate+up N = 2 x 4352 = 8704 from K = 5120, down N = 5120 from K = 4352.

@dataclass(frozen=True)
class DenseWorkload:
    name: str
    index: int   # seed family
    M: int       # token rows
    N: int       # output channels
    K: int       # reduction length


DENSE_WORKLOADS = {
    w.name: w
    for w in [
        DenseWorkload("dense_gate_up_m16", 50, 16, 8704, 5120),
        DenseWorkload("dense_down_m16", 51, 16, 5120, 4352),
        DenseWorkload("dense_small", 52, 8, 512, 256),
    ]
}


def dense_with_tokens(wl: DenseWorkload, M: int) -> DenseWorkload:
    return DenseWorkload(wl.name, wl.index, M, wl.N, wl.K)


def dense_weight(wl: DenseWorkload) -> np.ndarray:
    """FP32 [N, K] ~ N(0, 0.02)."""
    r = np.random.Generator(np.random.PCG64(np.random.SeedSequence([1000 * wl.index + _W13, 0])))
    return r.standard_normal((wl.N, wl.K), dtype=np.float32) * np.float32(0.02)


def dense_activations(wl: DenseWorkload, variant: int = 0) -> np.ndarray:
    """x: FP16 [M, K] ~ N(0, 1)."""
    r = np.random.Generator(np.random.PCG64(np.random.SeedSequence([1000 * wl.index + _X, variant])))
    return r.standard_normal((wl.M, wl.K), dtype=np.float32).astype(np.float16)


def random_ids(wl: Workload, variant: int = 0) -> np.ndarray:
    """Random distinct expert ids per token, int32 [M, k] (for plan tests)."""
    r = _rng(wl, 20, variant)
    out = np.empty((wl.M, wl.k), np.int32)
    for t in range(wl.M):
        out[t] = r.choice(wl.E, size=wl.k, replace=False)
    return out
