"""Seeded synthetic inputs for the Q4_K MoE layer (shared by tests and the benchmark).

This module only draws random numbers: it holds none of the layer's
arithmetic (no Q4_K packing, no GEMV, no activation, no combine). Both the CUDA
path and the CPU oracle consume what it produces.

Recipes (one independent numpy stream per named input, seeded from a base
seed and the input's name):
  * weights: fp32 N(0, 0.02) per expert matrix, quantized to Q4_K by the caller;
  * activations (h_post, h_mid), shared-gate logits: fp32 N(0, 1);
  * ids, "uniform": every token draws top_k distinct experts uniformly
    (partial Fisher-Yates);
  * ids, "zipf": expert e has probability proportional to 1/(e+1)^s
    (rank = id); a token draws top_k distinct experts by weighted sampling
    without replacement (a repeated draw is redrawn);
  * routing weights: softmax over the top_k slots of N(0, 1) logits;
  * router weights: N(0, 1/hidden) stored as bf16 (round to nearest even), so the
    gate logits of N(0, 1) activations are about N(0, 1); correction biases
    uniform in [-0.05, 0.05]; norm weights 1 + N(0, 0.1) in bf16.
"""
from __future__ import annotations

import zlib

import numpy as np


def _stream(seed: int, name: str, *extra: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), zlib.crc32(name.encode()), *[int(x) for x in extra]])


def normal(seed: int, name: str, shape, std: float = 1.0, *extra: int) -> np.ndarray:
    g = _stream(seed, name, *extra)
    return (g.standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def expert_weights(seed: int, proj: str, expert: int, n: int, k: int, std: float = 0.02) -> np.ndarray:
    """fp32 [n, k] N(0, std) weights of one expert's projection (proj in gate/up/down/...)."""
    return normal(seed, "w_" + proj, (n, k), std, expert)


def to_bf16_bits(x) -> np.ndarray:
    """uint16 bf16 bit patterns of float32 values, rounded to nearest even (data conversion)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_normal(seed: int, name: str, shape, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    """uint16 bf16 bits of mean + N(0, std) draws."""
    return to_bf16_bits(normal(seed, name, shape, std) + np.float32(mean))


def uniform(seed: int, name: str, shape, lo: float, hi: float) -> np.ndarray:
    return _stream(seed, name).uniform(lo, hi, size=shape).astype(np.float32)


def ids_uniform_distinct(seed: int, m: int, top_k: int, num_experts: int, name: str = "ids") -> np.ndarray:
    g = _stream(seed, name)
    out = np.empty((m, top_k), np.int32)
    for t in range(m):
        pool = np.arange(num_experts)
        for s in range(top_k):  # partial Fisher-Yates
            j = int(g.integers(s, num_experts))
            pool[s], pool[j] = pool[j], pool[s]
        out[t] = pool[:top_k]
    return out.reshape(-1)


def ids_zipf_distinct(seed: int, m: int, top_k: int, num_experts: int, s: float = 1.1,
                      name: str = "ids") -> np.ndarray:
    g = _stream(seed, name)
    p = 1.0 / np.power(np.arange(1, num_experts + 1, dtype=np.float64), s)
    cdf = np.cumsum(p / p.sum())
    out = np.empty((m, top_k), np.int32)
    for t in range(m):
        chosen: list[int] = []
        while len(chosen) < top_k:
            e = int(np.searchsorted(cdf, g.random(), side="right"))
            e = min(e, num_experts - 1)
            if e not in chosen:
                chosen.append(e)
        out[t] = chosen
    return out.reshape(-1)


def routing_weights(seed: int, m: int, top_k: int, name: str = "route") -> np.ndarray:
    z = _stream(seed, name).standard_normal((m, top_k))
    z = np.exp(z - z.max(axis=1, keepdims=True))
    return (z / z.sum(axis=1, keepdims=True)).astype(np.float32).reshape(-1)


def make_ids(seed: int, dist: str, m: int, top_k: int, num_experts: int, name: str = "ids") -> np.ndarray:
    if dist == "uniform":
        return ids_uniform_distinct(seed, m, top_k, num_experts, name)
    if dist == "zipf":
        return ids_zipf_distinct(seed, m, top_k, num_experts, 1.1, name)
    raise ValueError(dist)
