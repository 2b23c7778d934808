"""Seeded synthetic inputs for the W4A16 MoE expert path.

This module only draws random inputs: uint4 weight codes, BF16 group scales,
BF16 activations and top-k routing.  It holds none of the method's
arithmetic (no dequantisation, no GEMM, no alignment), so the CUDA path and
the CPU oracle can both consume its arrays without sharing any code.

Recipe (the same for every workload):

* weight codes: uniform uint32 words, each word being 8 uniform uint4 codes,
  stored as int32 ``[E, N, K/8]``; element ``k`` of a row sits in word
  ``k // 8`` at bits ``4*(k % 8) .. +3`` (low nibble first);
* scales: uniform in ``[0.005, 0.02]``, rounded to BF16 (round to nearest
  even), ``[E, N, K/32]``;
* activations: BF16 of N(0, 1) draws, ``[T, H]``;
* routing, softmax kind: router logits N(0, 1) over all global experts,
  ``softmax``, the top-k probabilities (ties to the lower expert id); the
  weights are the selected probabilities, not renormalised;
* routing, Zipf kind: Gumbel-top-k over log-weights ``-s*ln(pi(e)+1)`` with
  ``pi`` a seeded permutation of the global experts (sampling without
  replacement proportional to a Zipf(s) law); the weights are the softmax of
  the perturbed logits at the selected experts;
* expert parallel slice: global ids outside the local range become ``-1``
  (a dropped slot); local ids are shifted to start at 0.

Seeds: weights ``100*cfg``, routing and activations ``1000*cfg + T`` (two
independent streams of that seed); the Zipf draw of the tensor-parallel
workload uses ``5000 + T``.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Sequence, Tuple

import numpy as np
import torch

GROUP = 32


@dataclass(frozen=True)
class MoEWorkload:
    """Shapes of one synthetic MoE layer (one rank of it)."""

    name: str
    cfg_id: int
    E: int            # experts held by this rank
    E_global: int     # experts the router chooses from
    top_k: int
    H: int            # hidden size (K of gate_up, N of down)
    I: int            # expert intermediate size per rank (N of gate_up is 2*I)
    tokens: Tuple[int, ...]
    routing: str = "softmax"          # "softmax" | "zipf"
    local_lo: int = 0                 # first global expert held by this rank
    empty_experts: Tuple[int, ...] = ()
    block_m: Optional[int] = None     # fixed block_m (None: the planner picks)
    zipf_s: float = 1.1
    routing_seed_base: Optional[int] = None

    @property
    def gate_up_shape(self):
        return (self.E, 2 * self.I, self.H)

    @property
    def down_shape(self):
        return (self.E, self.H, self.I)

    def weight_seed(self) -> int:
        return 100 * self.cfg_id

    def routing_seed(self, T: int) -> int:
        base = self.routing_seed_base if self.routing_seed_base is not None else 1000 * self.cfg_id
        return base + T


WORKLOADS = {
    # Tiny layer: E=8, top-2 of softmax(N(0,1)) with expert 7 forced empty,
    # hidden 256, gate_up [8,512,256], down [8,256,256], block_m 16.
    "tiny": MoEWorkload("tiny", 1, 8, 8, 2, 256, 256, (16,), empty_experts=(7,), block_m=16),
    # Qwen3-30B-A3B-shaped experts: 128 experts, top-8, hidden 2048,
    # gate_up [128,1536,2048], down [128,2048,768].
    "qwen3_30b_a3b": MoEWorkload("qwen3_30b_a3b", 2, 128, 128, 8, 2048, 768, (1, 8, 64, 512, 4096)),
    # Kimi-K2-shaped expert-parallel rank (48 of 384 experts), decode sweep.
    "kimi_k2_ep8_decode": MoEWorkload("kimi_k2_ep8_decode", 3, 48, 384, 8, 7168, 2048,
                                      (1, 16, 64, 128, 256)),
    # Same rank, prefill sweep with Zipf(1.1)-skewed routing.
    "kimi_k2_ep8_prefill": MoEWorkload("kimi_k2_ep8_prefill", 4, 48, 384, 8, 7168, 2048,
                                       (2048, 4096, 8192, 16384), routing="zipf"),
    # Kimi-K2-shaped tensor-parallel rank: all 384 experts, intermediate 256.
    "kimi_k2_tp8": MoEWorkload("kimi_k2_tp8", 5, 384, 384, 8, 7168, 256, (1, 32, 256, 1024, 8192)),
    "kimi_k2_tp8_zipf": MoEWorkload("kimi_k2_tp8_zipf", 5, 384, 384, 8, 7168, 256,
                                    (1, 32, 256, 1024, 8192), routing="zipf", routing_seed_base=5000),
}


def draw_weights(E: int, N: int, K: int, seed: int, group: int = GROUP):
    """uint4 codes packed 8 per int32 along K, and BF16 scales per group of K.

    Returns ``(qweight int32 [E, N, K/8], scales bf16 [E, N, K/group])`` on the CPU.
    """
    if K % 8 or K % group:
        raise ValueError("K must be a multiple of 8 and of the group size")
    rng = np.random.default_rng([seed, 0])
    words = rng.integers(0, 2 ** 32, size=(E, N, K // 8), dtype=np.uint32)
    qweight = torch.from_numpy(words.view(np.int32))
    rng_s = np.random.default_rng([seed, 1])
    s = rng_s.uniform(0.005, 0.02, size=(E, N, K // group)).astype(np.float32)
    scales = torch.from_numpy(s).to(torch.bfloat16)
    return qweight, scales


def draw_nvfp4_weights(E: int, N: int, K: int, seed: int):
    """NVFP4 weights: E2M1 codes two per byte along K (element 2j in the low nibble), uniform
    over all 256 byte values, and one positive E4M3 scale byte per 16 K elements with an
    exponent field of 1 or 2 and a uniform mantissa (scales in [2^-6, 2^-4 * 15/16]).

    Returns ``(codes uint8 [E, N, K/2], scales uint8 [E, N, K/16])`` on the CPU.
    """
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    rng = np.random.default_rng([seed, 3])
    codes = rng.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    rng_s = np.random.default_rng([seed, 4])
    exp_field = rng_s.integers(1, 3, size=(E, N, K // 16), dtype=np.uint8)
    mant = rng_s.integers(0, 8, size=(E, N, K // 16), dtype=np.uint8)
    scales = (exp_field << 3) | mant
    return torch.from_numpy(codes), torch.from_numpy(scales)


def draw_activations(T: int, H: int, seed: int) -> torch.Tensor:
    """BF16 of N(0,1) draws, ``[T, H]`` on the CPU."""
    rng = np.random.default_rng([seed, 2])
    x = rng.standard_normal((T, H), dtype=np.float32)
    return torch.from_numpy(x).to(torch.bfloat16)


def _softmax_rows(z: np.ndarray) -> np.ndarray:
    m = np.max(z, axis=1, keepdims=True)
    p = np.exp(z - m)
    return p / np.sum(p, axis=1, keepdims=True)


def draw_routing(T: int, E_global: int, top_k: int, seed: int, kind: str = "softmax",
                 local_lo: int = 0, E_local: Optional[int] = None,
                 empty_experts: Sequence[int] = (), zipf_s: float = 1.1):
    """Top-k routing draw.

    Returns ``(topk_ids int32 [T, k], topk_weights float32 [T, k])``; ids are
    local expert ids, or -1 for a slot whose expert lives on another rank.
    """
    E_local = E_global if E_local is None else E_local
    rng = np.random.default_rng([seed, 1])
    if kind == "softmax":
        logits = rng.standard_normal((T, E_global))
        if len(empty_experts):
            logits[:, list(empty_experts)] = -np.inf
        score = logits
        probs = _softmax_rows(logits)
    elif kind == "zipf":
        rank = rng.permutation(E_global)
        base = -zipf_s * np.log(rank + 1.0)
        score = base[None, :] + rng.gumbel(size=(T, E_global))
        if len(empty_experts):
            score[:, list(empty_experts)] = -np.inf
        probs = _softmax_rows(score)
    else:
        raise ValueError(f"unknown routing kind {kind!r}")
    # descending score, ties to the lower expert id (stable sort of -score)
    order = np.argsort(-score, axis=1, kind="stable")[:, :top_k]
    weights = np.take_along_axis(probs, order, axis=1).astype(np.float32)
    ids = order.astype(np.int64)
    local = (ids >= local_lo) & (ids < local_lo + E_local)
    ids = np.where(local, ids - local_lo, -1).astype(np.int32)
    return torch.from_numpy(ids), torch.from_numpy(weights)


@dataclass
class LayerInputs:
    """One seeded draw of a whole layer's inputs, on the CPU."""

    wl: MoEWorkload
    T: int
    x: torch.Tensor
    topk_ids: torch.Tensor
    topk_weights: torch.Tensor
    w13_q: torch.Tensor = field(repr=False)
    w13_s: torch.Tensor = field(repr=False)
    w2_q: torch.Tensor = field(repr=False)
    w2_s: torch.Tensor = field(repr=False)


def draw_layer_weights(wl: MoEWorkload):
    seed = wl.weight_seed()
    w13_q, w13_s = draw_weights(wl.E, 2 * wl.I, wl.H, seed)
    w2_q, w2_s = draw_weights(wl.E, wl.H, wl.I, seed + 1)
    return w13_q, w13_s, w2_q, w2_s


def draw_layer_routing(wl: MoEWorkload, T: int):
    seed = wl.routing_seed(T)
    ids, w = draw_routing(T, wl.E_global, wl.top_k, seed, wl.routing, wl.local_lo, wl.E,
                          wl.empty_experts, wl.zipf_s)
    x = draw_activations(T, wl.H, seed)
    return x, ids, w


def draw_layer(wl: MoEWorkload, T: int, weights=None) -> LayerInputs:
    if weights is None:
        weights = draw_layer_weights(wl)
    x, ids, w = draw_layer_routing(wl, T)
    return LayerInputs(wl, T, x, ids, w, *weights)
