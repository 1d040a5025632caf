"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module only draws random numbers and packs them as bf16 bit patterns.
It holds none of the method's arithmetic (no gather, no GEMM, no reduction, no
routing bookkeeping), so both sides of a parity test can take their inputs
from here without sharing any computation.

Conventions
-----------
* Every tensor is drawn from its own ``numpy.random.Generator(PCG64(seed))``.
  Seeds: shard r -> base+r; B (or B_r) -> base+1000(+r); expert weight W_e ->
  base+2000+e; routing -> base+3000; MoE down side -> base+4000..6000;
  attention Q -> base+7000, K_r -> base+8000+r, V_r -> base+9000+r.
  numpy's PCG64 bit stream is stable across
  platforms, so x86 and aarch64 hosts draw identical inputs.
* Values are drawn in float32 and rounded to bfloat16 with round-to-nearest-even
  (the packing step of the bfloat16 storage format: keep the top 16 bits of the
  IEEE binary32 pattern after adding the tie-to-even bias).  Arrays are returned
  as ``uint16`` bit patterns; ``to_torch_bf16`` reinterprets them.
* MoE routing: top-k distinct experts per token drawn from a finite Zipf law
  p(e) proportional to 1/(e+1)^s over e = 0..E-1, without replacement, slot
  order = draw order.  Sampling without replacement with successive
  renormalisation is drawn with the Gumbel-top-k construction (the k largest of
  log p(e) + Gumbel noise), which has exactly that law.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "CONFIGS", "bf16_bits_from_f32", "uniform_bf16", "normal_bf16",
    "ag_gemm_inputs", "gemm_rs_inputs", "moe_inputs", "zipf_topk",
    "to_torch_bf16", "moe_down_inputs", "ag_attention_inputs",
]

# The five workloads (shapes, value distributions).  Names describe the workload.
CONFIGS = {
    "ag_tiny": dict(kind="ag", R=2, M_shard=128, K=512, N=256, dist="uniform"),
    "ag_llm": dict(kind="ag", R=8, M_shard=1024, K=4096, N=1792, dist="normal"),
    "rs_llm": dict(kind="rs", R=8, M=8192, K_r=1792, N=4096),
    "moe_llm": dict(kind="moe", R=8, T_r=1024, H=4096, N=1408, E=32, topk=2, zipf_s=1.2),
    # AG sweep: total M in {1024..16384}, K=8192, N=1024, R in {2,4,8}
    "ag_sweep": dict(kind="ag_sweep", R=(2, 4, 8), M=(1024, 2048, 4096, 8192, 16384), K=8192, N=1024),
}


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Pack float32 values as bfloat16 bit patterns (round to nearest, ties to even).

    Finite inputs only (the generators never draw inf/NaN)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + bias) >> np.uint64(16)).astype(np.uint16)


def uniform_bf16(shape, seed: int, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    x = _rng(seed).uniform(lo, hi, size=shape).astype(np.float32)
    return bf16_bits_from_f32(x)


def normal_bf16(shape, seed: int, std: float = 1.0) -> np.ndarray:
    x = _rng(seed).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return bf16_bits_from_f32(x)


def ag_gemm_inputs(R: int, M_shard: int, K: int, N: int, dist: str = "normal", seed: int = 0):
    """A_r [M_shard, K] for r in 0..R-1 and B [K, N], as bf16 bit arrays.

    dist="uniform": U[-1,1) for both; dist="normal": A ~ N(0,1), B ~ N(0,0.02)."""
    if dist == "uniform":
        A = [uniform_bf16((M_shard, K), seed + r) for r in range(R)]
        B = uniform_bf16((K, N), seed + 1000)
    elif dist == "normal":
        A = [normal_bf16((M_shard, K), seed + r, 1.0) for r in range(R)]
        B = normal_bf16((K, N), seed + 1000, 0.02)
    else:
        raise ValueError(dist)
    return A, B


def gemm_rs_inputs(R: int, M: int, K_r: int, N: int, seed: int = 0):
    """Per-rank A_r [M, K_r] ~ N(0,1) and B_r [K_r, N] ~ N(0,0.02), bf16 bits."""
    A = [normal_bf16((M, K_r), seed + r, 1.0) for r in range(R)]
    B = [normal_bf16((K_r, N), seed + 1000 + r, 0.02) for r in range(R)]
    return A, B


def zipf_topk(T: int, E: int, k: int, s: float, seed: int) -> np.ndarray:
    """topk_ids [T, k] int32: k distinct experts per token, finite Zipf(s) law."""
    if k > E:
        raise ValueError("k > E")
    logp = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    u = _rng(seed).random(size=(T, E))
    u = np.clip(u, 1e-300, 1.0 - 1e-16)
    keys = logp[None, :] - np.log(-np.log(u))
    order = np.argsort(-keys, axis=1, kind="stable")
    return np.ascontiguousarray(order[:, :k].astype(np.int32))


def moe_inputs(R: int, T_r: int, H: int, N: int, E: int, topk: int, zipf_s: float = 1.2,
               seed: int = 0, with_weights: bool = True):
    """Token shards X_r [T_r, H] ~ N(0,1), routing [R*T_r, topk], weights W_e [H, N] ~ N(0,0.02)."""
    X = [normal_bf16((T_r, H), seed + r, 1.0) for r in range(R)]
    topk_ids = zipf_topk(R * T_r, E, topk, zipf_s, seed + 3000)
    W = [normal_bf16((H, N), seed + 2000 + e, 0.02) for e in range(E)] if with_weights else None
    return X, topk_ids, W


def to_torch_bf16(bits: np.ndarray):
    """Reinterpret a uint16 bit array as a torch.bfloat16 CPU tensor (no copy of values)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def moe_down_inputs(R: int, T_r: int, topk: int, E: int, I_r: int, Hd: int, seed: int = 0):
    """The down-projection side of the MoE layer: per-rank intermediate activations
    H_r [R*T_r*topk, I_r] ~ N(0,1) in expert-sorted row order, per-rank weights
    W2_r [E*I_r, Hd] ~ N(0,0.02) (expert e's slice at rows e*I_r), bf16 bits, and
    gate weights [R*T_r, topk] float32, uniform(0,1) normalised to sum 1 per token."""
    P = R * T_r * topk
    H = [normal_bf16((P, I_r), seed + 4000 + r, 1.0) for r in range(R)]
    W2 = [normal_bf16((E * I_r, Hd), seed + 5000 + r, 0.02) for r in range(R)]
    g = np.random.Generator(np.random.PCG64(seed + 6000)).uniform(0.0, 1.0, (R * T_r, topk)).astype(np.float32)
    gates = (g / g.sum(axis=1, keepdims=True)).astype(np.float32)
    return H, W2, gates


def ag_attention_inputs(R: int, S_shard: int, H: int, H_kv: int, D: int = 128, seed: int = 0):
    """Sequence-parallel attention inputs: this rank's queries Q [S_shard, H, D]
    and every rank's keys and values K_r, V_r [S_shard, H_kv, D], all N(0,1)
    bf16 bits (unit-variance activations after the projections).  Seeds: Q ->
    base+7000, K_r -> base+8000+r, V_r -> base+9000+r."""
    Q = normal_bf16((S_shard, H, D), seed + 7000)
    K = [normal_bf16((S_shard, H_kv, D), seed + 8000 + r) for r in range(R)]
    V = [normal_bf16((S_shard, H_kv, D), seed + 9000 + r) for r in range(R)]
    return Q, K, V
