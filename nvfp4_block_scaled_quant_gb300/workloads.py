"""Seeded synthetic inputs shaped like the MoE workloads of a large MoE LLM.

This module only draws random numbers: it holds no quantisation, GEMM or
routing arithmetic of the method, and both the CUDA path and the CPU oracle
take their inputs from it.  Every generator is a torch.Generator seeded from
an integer, on the device the caller names (draws on 'cuda' and 'cpu' differ,
so a test that compares devices draws once and copies).

Recipes
-------
* activations: bf16 N(0, 1); with ``outliers`` 1 % of the channels (a seeded
  permutation prefix) are scaled by 20;
* weights: bf16 N(0, 0.02), one generator per expert matrix;
* routing ``softmax``: logits N(0, 1) over E experts, top-k by value, weights
  the softmax renormalised over the k chosen;
* routing ``uniform``: k distinct experts per token (seeded permutation
  prefix), weights softmax of N(0, 1) over the k slots;
* routing ``zipf``: k distinct experts per token drawn by Gumbel-top-k from
  p_e proportional to rank(e)^-s (rank one seeded permutation of the ids per
  workload, so the popular experts stay popular from chunk to chunk), weights
  softmax of N(0, 1) over the k slots.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Tuple

import torch

WEIGHT_STD = 0.02
OUTLIER_FRACTION = 0.01
OUTLIER_GAIN = 20.0


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def activations(T: int, H: int, seed: int, device="cpu", outliers: bool = False) -> torch.Tensor:
    g = _gen(seed, device)
    x = torch.randn(T, H, generator=g, device=device, dtype=torch.float32)
    if outliers:
        n = max(1, int(round(OUTLIER_FRACTION * H)))
        cols = torch.randperm(H, generator=g, device=device)[:n]
        x[:, cols] *= OUTLIER_GAIN
    return x.to(torch.bfloat16)


def weight(N: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return (torch.randn(N, K, generator=g, device=device, dtype=torch.float32) * WEIGHT_STD).to(torch.bfloat16)


def expert_seeds(base: int, e: int) -> Tuple[int, int]:
    """Seeds of expert e's (w13, w2) matrices; the shared expert uses e = E."""
    return base * 4099 + 2 * e, base * 4099 + 2 * e + 1


def routing_softmax(T: int, E: int, k: int, seed: int, device="cpu"):
    g = _gen(seed, device)
    logits = torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    p = torch.softmax(logits, dim=-1)
    w, ids = torch.topk(p, k, dim=-1)
    w = w / w.sum(dim=-1, keepdim=True)
    return ids.to(torch.int32).contiguous(), w.contiguous()


def _slot_weights(T: int, k: int, g, device) -> torch.Tensor:
    return torch.softmax(torch.randn(T, k, generator=g, device=device, dtype=torch.float32), dim=-1).contiguous()


def routing_uniform(T: int, E: int, k: int, seed: int, device="cpu"):
    g = _gen(seed, device)
    keys = torch.rand(T, E, generator=g, device=device)
    ids = torch.argsort(keys, dim=-1)[:, :k]
    return ids.to(torch.int32).contiguous(), _slot_weights(T, k, g, device)


ZIPF_RANK_SEED = 4242  # one expert-popularity ranking per workload, shared by all its chunks


def routing_zipf(T: int, E: int, k: int, seed: int, device="cpu", s: float = 1.1):
    rank = torch.randperm(E, generator=_gen(ZIPF_RANK_SEED, device), device=device).to(torch.float64) + 1.0
    g = _gen(seed, device)
    logp = -s * torch.log(rank)
    u = torch.rand(T, E, generator=g, device=device, dtype=torch.float64).clamp_min(1e-300)
    gumbel = -torch.log(-torch.log(u))
    ids = torch.topk(logp[None, :] + gumbel, k, dim=-1).indices
    return ids.to(torch.int32).contiguous(), _slot_weights(T, k, g, device)


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    topk: int
    shared: bool
    routing: str       # softmax | uniform | zipf
    outliers: bool
    chunks: int = 1    # sequential calls of T tokens (prefill)


# The workloads (token counts, widths, expert counts) of the five configurations.
TINY = MoEConfig("tiny_moe_T16_H256_I128_E8_k2", 16, 256, 128, 8, 2, False, "softmax", False)
TINY_SHARED = MoEConfig("tiny_moe_shared_T16_H256_I128_E8_k2", 16, 256, 128, 8, 2, True, "softmax", False)
DECODE = {T: MoEConfig(f"decode_moe_T{T}_H7168_I2048_E384_k8", T, 7168, 2048, 384, 8, True, "uniform", False)
          for T in (1, 8, 64)}
PREFILL = MoEConfig("prefill_moe_32x128_H7168_I2048_E384_k8_zipf1.1", 128, 7168, 2048, 384, 8, True, "zipf", True,
                    chunks=32)
DENSE_LINEAR = {M: (M, 1536, 16384) for M in (1, 32, 128)}   # (M, K, N), outlier activations
DENSE_GEMM = {M: (M, 7168, 7168) for M in (1024, 4096, 16384)}


def routing(cfg: MoEConfig, seed: int, device="cpu"):
    fn = {"softmax": routing_softmax, "uniform": routing_uniform, "zipf": routing_zipf}[cfg.routing]
    return fn(cfg.T, cfg.E, cfg.topk, seed, device)


# Seeds of the timed workloads, shared by the benchmark and the parity tests that
# replay them.
BENCH_WEIGHT_SEED = 2024


def prefill_chunk(c: int, device="cpu"):
    """Chunk c (0..31) of the prefill workload: x (128, 7168) with outlier channels, zipf top-8 routing."""
    cfg = PREFILL
    x = activations(cfg.T, cfg.H, seed=700_000 + c, device=device, outliers=cfg.outliers)
    ids, w = routing(cfg, seed=800_000 + c, device=device)
    return x, ids, w


def decode_step(T: int, step: int = 0, device="cpu"):
    cfg = DECODE[T]
    x = activations(T, cfg.H, seed=900_000 + 100 * T + step, device=device)
    ids, w = routing(cfg, seed=950_000 + 100 * T + step, device=device)
    return x, ids, w


PREFILL_WHOLE = MoEConfig("prefill_whole_moe_T4096_H7168_I2048_E384_k8_zipf1.1", 4096, 7168, 2048, 384, 8, True,
                          "zipf", True)


def prefill_whole(device="cpu"):
    """The 32 prefill chunks' tokens and routings in one 4096-token call."""
    parts = [prefill_chunk(c, device) for c in range(PREFILL.chunks)]
    return (torch.cat([p[0] for p in parts]).contiguous(), torch.cat([p[1] for p in parts]).contiguous(),
            torch.cat([p[2] for p in parts]).contiguous())


# Fixed-group linear (grouped o-projection): 8 groups of 4096 inputs each; the output width per
# group is not printed on the pages, 1024 is taken (a multiple of the 128-wide tile).
GROUPED_LINEAR = {M: (M, 8, 4096, 1024) for M in (1, 128)}   # (M, G, K, N)


RMSNORM_EPS = 1e-6


def norm_weight(K: int, seed: int, device="cpu") -> torch.Tensor:
    """RMSNorm gain: bf16 1 + 0.1 N(0, 1)."""
    g = _gen(seed, device)
    return (1.0 + 0.1 * torch.randn(K, generator=g, device=device)).to(torch.bfloat16)


# Router gate of the 384-expert layer: gate weight (E, H) bf16 N(0, 0.02) stored as NVFP4.
ROUTER = {T: (T, 7168, 384, 8) for T in (1, 128)}   # (T, H, E, topk)
ROUTER_WEIGHT_SEED = 31337
