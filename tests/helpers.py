"""Shared test helpers: oracle-side expert construction and the parity checks."""

from __future__ import annotations

import numpy as np
import torch

from nvfp4_block_scaled_quant_gb300 import workloads
from oracle import nvfp4_oracle as O

# Parity bar for GEMM / MoE outputs on identical dequantised operands:
# |y - y_ref| <= REL * |y_ref| + ABS_RMS * rms(y_ref) element-wise, and cosine >= COS.
REL = 1e-2
ABS_RMS = 1e-3
COS = 0.9999


def assert_parity(got, ref, rel=REL, abs_rms=ABS_RMS, cos_min=COS, what="output"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    err = np.abs(got - ref)
    bound = rel * np.abs(ref) + abs_rms * rms
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements outside the bound; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} bound {bound[i]!r}")
    c = O.cosine(got, ref)
    assert c >= cos_min, f"{what}: cosine {c}"
    return c


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def oracle_expert_fn(base_seed: int, H: int, I: int, device):
    """Oracle-side experts: regenerate each bf16 matrix from its seed and quantise it in the oracle."""
    cache = {}

    def get(e: int) -> O.Expert:
        if e not in cache:
            s13, s2 = workloads.expert_seeds(base_seed, e)
            q13 = O.quantize(workloads.weight(2 * I, H, s13, device).float().cpu().numpy())
            q2 = O.quantize(workloads.weight(H, I, s2, device).float().cpu().numpy())
            cache[e] = O.Expert(q13.codes, q13.sf, q13.gs, q2.codes, q2.sf, q2.gs)
        return cache[e]

    return get


def unswizzle(buf: torch.Tensor, rows: int, K: int) -> np.ndarray:
    return O.unswizzle_sf(buf.detach().cpu().numpy().ravel(), rows, K)


def unpack(codes: torch.Tensor) -> np.ndarray:
    return O.unpack_codes(codes.detach().cpu().numpy())
