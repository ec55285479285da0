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


class OracleExperts:
    """Oracle-side experts: regenerate each bf16 matrix from its seed (drawn on ``device``, as the
    library-side weights are) and quantise it in the oracle.  Picklable (the cache stays behind),
    so the oracle's per-expert jobs can run in a spawned process pool."""

    def __init__(self, base_seed: int, H: int, I: int, device):
        self.base_seed, self.H, self.I, self.device = base_seed, H, I, str(device)
        self.cache = {}

    def __getstate__(self):
        return {"base_seed": self.base_seed, "H": self.H, "I": self.I, "device": self.device}

    def __setstate__(self, st):
        self.__dict__.update(st)
        self.cache = {}

    def __call__(self, e: int) -> O.Expert:
        if e not in self.cache:
            s13, s2 = workloads.expert_seeds(self.base_seed, e)
            q13 = O.quantize(workloads.weight(2 * self.I, self.H, s13, self.device).float().cpu().numpy())
            q2 = O.quantize(workloads.weight(self.H, self.I, s2, self.device).float().cpu().numpy())
            self.cache[e] = O.Expert(q13.codes, q13.sf, q13.gs, q2.codes, q2.sf, q2.gs)
        return self.cache[e]


def oracle_expert_fn(base_seed: int, H: int, I: int, device) -> OracleExperts:
    return OracleExperts(base_seed, H, I, device)


def oracle_pool(workers: int = 16):
    """A spawned process pool for the oracle's per-expert jobs (each worker single-threaded BLAS).
    Spawned, not forked: the parent already holds a CUDA context."""
    import multiprocessing as mp
    import os

    n = max(1, min(workers, os.cpu_count() or 1))
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    os.environ.update({k: "1" for k in keys})  # the children inherit the environment at spawn
    try:
        return mp.get_context("spawn").Pool(n)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def unswizzle(buf: torch.Tensor, rows: int, K: int) -> np.ndarray:
    return O.unswizzle_sf(buf.detach().cpu().numpy().ravel(), rows, K)


def unpack(codes: torch.Tensor) -> np.ndarray:
    return O.unpack_codes(codes.detach().cpu().numpy())
