"""Load-time helpers: NVFP4 checkpoints made from bf16 matrices and prepared MoE/linear weights.

Everything runs through the library (quantize + prepare kernels).  A bf16
weight quantises with its own global scale ws2 = amax/2688 into the
checkpoint layout (codes (N, K/2), row-major scales (N, K/16)), which the
prepare step turns into the device layout; nothing here runs per token.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Tuple

import torch

from . import ops, workloads


def quantize_weight(w: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """bf16 (N, K) -> checkpoint codes (N, K/2), row-major E4M3 scales (N, K/16), ws2 (1,)."""
    return ops.quantize_act(w, gs=None, sf_layout="linear")


@dataclass
class DenseWeight:
    N: int
    K: int
    w: torch.Tensor       # prepared codes (N, K/2)
    sf: torch.Tensor      # swizzled scales
    ws2: torch.Tensor     # (1,) fp32


def make_dense_weight(N: int, K: int, seed: int, device) -> DenseWeight:
    wb = workloads.weight(N, K, seed, device)
    q, sf, ws2 = quantize_weight(wb)
    wp, sfp = ops.prepare_weights(q, sf, N, K, interleave_w13=False)
    return DenseWeight(N, K, wp, sfp, ws2)


def make_moe_weights(E: int, H: int, I: int, base_seed: int, device, shared: bool = True) -> ops.MoEWeights:
    """Synthetic experts: bf16 N(0, 0.02) per matrix, quantised and prepared on the device."""
    dev = torch.device(device)
    w13_ck = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=dev)
    w13_sf = torch.empty(E, 2 * I, H // 16, dtype=torch.uint8, device=dev)
    w2_ck = torch.empty(E, H, I // 2, dtype=torch.uint8, device=dev)
    w2_sf = torch.empty(E, H, I // 16, dtype=torch.uint8, device=dev)
    w13_ws2 = torch.empty(E, dtype=torch.float32, device=dev)
    w2_ws2 = torch.empty(E, dtype=torch.float32, device=dev)
    for e in range(E):
        s13, s2 = workloads.expert_seeds(base_seed, e)
        q, sf, g = quantize_weight(workloads.weight(2 * I, H, s13, dev))
        w13_ck[e].copy_(q)
        w13_sf[e].copy_(sf.view(2 * I, H // 16))
        w13_ws2[e : e + 1].copy_(g)
        q, sf, g = quantize_weight(workloads.weight(H, I, s2, dev))
        w2_ck[e].copy_(q)
        w2_sf[e].copy_(sf.view(H, I // 16))
        w2_ws2[e : e + 1].copy_(g)
    w13, w13_sfp = ops.prepare_weights(w13_ck, w13_sf, 2 * I, H, interleave_w13=True)
    del w13_ck, w13_sf
    w2, w2_sfp = ops.prepare_weights(w2_ck, w2_sf, H, I, interleave_w13=False)
    del w2_ck, w2_sf
    W = ops.MoEWeights(E, H, I, w13, w13_sfp, w13_ws2, w2, w2_sfp, w2_ws2)
    if shared:
        s13, s2 = workloads.expert_seeds(base_seed, E)
        q13, sf13, g13 = quantize_weight(workloads.weight(2 * I, H, s13, dev))
        q2, sf2, g2 = quantize_weight(workloads.weight(H, I, s2, dev))
        W.sh_w13, W.sh_w13_sf = ops.prepare_weights(q13, sf13, 2 * I, H, interleave_w13=True)
        W.sh_w2, W.sh_w2_sf = ops.prepare_weights(q2, sf2, H, I, interleave_w13=False)
        W.sh_ws2 = torch.cat([g13, g2]).contiguous()
    return W


@dataclass
class GroupedWeight:
    G: int
    N: int
    K: int
    w: torch.Tensor       # prepared codes (G, N, K/2)
    sf: torch.Tensor      # G swizzled scale blocks
    ws2: torch.Tensor     # (G,) fp32


def make_grouped_weight(G: int, N: int, K: int, seed: int, device) -> GroupedWeight:
    """G independent bf16 N(0, 0.02) matrices (N, K), each quantised with its own ws2, then prepared."""
    dev = torch.device(device)
    ck = torch.empty(G, N, K // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty(G, N, K // 16, dtype=torch.uint8, device=dev)
    ws2 = torch.empty(G, dtype=torch.float32, device=dev)
    for g in range(G):
        q, s, w2 = quantize_weight(workloads.weight(N, K, seed * 1009 + g, dev))
        ck[g].copy_(q)
        sf[g].copy_(s.view(N, K // 16))
        ws2[g:g + 1].copy_(w2)
    wp, sfp = ops.prepare_weights(ck, sf, N, K)
    return GroupedWeight(G, N, K, wp, sfp, ws2)
