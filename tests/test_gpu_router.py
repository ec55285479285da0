"""Router gate on the GPU against the oracle.

The prepared gate weight (NVFP4 -> bf16 -> FP8-E4M3 round trip -> bf16) is bit-exact; logits
meet the GEMM bound; ids match exactly for every token whose oracle probabilities are separated
by more than 1e-5 (relative) around the top-k boundary and between chosen experts, and the
renormalised weights agree to 1e-4.  The router's output also drives the routed MoE end to end.
"""

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_quant_gb300 import model, ops, workloads
from oracle import nvfp4_oracle as O
from tests.helpers import assert_parity, bf16_to_np, oracle_expert_fn

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _gate(E, H, seed):
    wb = workloads.weight(E, H, seed, DEV)
    q, sf, ws2 = model.quantize_weight(wb)
    wg = ops.router_prepare(q, sf, ws2, E, H)
    torch.cuda.synchronize()
    wq = O.quantize(wb.float().cpu().numpy())
    ref = O.router_weight(wq.codes, wq.sf, wq.gs)
    np.testing.assert_array_equal(bf16_to_np(wg), ref)  # bit-exact
    return wg, ref


def _check_router(x, wg, wg_ref, k):
    ids, w, logits = ops.router(x.to(DEV), wg, k, want_logits=True)
    torch.cuda.synchronize()
    rid, rw, p = O.router(x.float().numpy(), wg_ref, k)
    lref = x.float().numpy().astype(np.float64) @ wg_ref.astype(np.float64).T
    assert_parity(logits.cpu().numpy(), lref, what="router logits")
    # fp32 logits over H terms are accurate to ~1e-6 relative; a token is "clear" when its top-k+1
    # probabilities are 1e-5 (relative) apart, and at most 1% of the tokens (rounded down) may not be
    ps = -np.sort(-p, axis=1)[:, : k + 1]
    gaps = (ps[:, :-1] - ps[:, 1:]) / ps[:, :-1]
    clear = (gaps > 1e-5).all(axis=1)
    assert clear.sum() >= int(np.floor(0.99 * len(clear))), f"{(~clear).sum()} of {len(clear)} tokens not clear"
    np.testing.assert_array_equal(ids.cpu().numpy()[clear], rid[clear])
    np.testing.assert_allclose(w.cpu().numpy()[clear], rw[clear], rtol=1e-4, atol=1e-7)
    np.testing.assert_allclose(w.cpu().numpy().sum(1), 1.0, rtol=1e-5)
    return ids, w


@pytest.mark.parametrize("T", sorted(workloads.ROUTER))
def test_router_workload(T):
    _, H, E, k = workloads.ROUTER[T]
    wg, ref = _gate(E, H, workloads.ROUTER_WEIGHT_SEED)
    x = workloads.activations(T, H, seed=40 + T, device="cpu")
    _check_router(x, wg, ref, k)


def test_router_small_shapes_and_ties():
    wg, ref = _gate(24, 256, 7)
    _check_router(workloads.activations(37, 256, seed=1, device="cpu"), wg, ref, 5)
    # all-zero tokens: uniform probabilities, ids 0..k-1 in order, equal weights
    ids, w, _ = ops.router(torch.zeros(3, 256, dtype=torch.bfloat16, device=DEV), wg, 4)
    torch.cuda.synchronize()
    assert ids.cpu().tolist() == [[0, 1, 2, 3]] * 3
    np.testing.assert_allclose(w.cpu().numpy(), 0.25, rtol=1e-6)


def test_router_drives_moe_end_to_end():
    """x -> router -> routed MoE (+ shared expert) against the oracle's router and MoE."""
    cfg = workloads.TINY_SHARED
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.topk
    wg, ref = _gate(E, H, 9)
    x = workloads.activations(T, H, seed=3, device="cpu")
    ids, w = _check_router(x, wg, ref, k)
    W = model.make_moe_weights(E, H, I, 109, DEV, shared=True)
    oe = oracle_expert_fn(109, H, I, DEV)
    a2 = np.full(E + 1, np.float32(0.004), np.float32)
    y, _ = ops.moe_forward(x.to(DEV), ids, w, W, torch.from_numpy(a2).to(DEV))
    torch.cuda.synchronize()
    rid, rw, _ = O.router(x.float().numpy(), ref, k)
    res = O.moe_forward(x.float().numpy(), rid, rw.astype(np.float32), oe, E, a2, shared=oe(E))
    assert O.cosine(bf16_to_np(y), res.y) > 0.999


def test_router_expert_count_not_multiple_of_4_and_unaligned_logits():
    """E not a multiple of 4 (the logits kernel's rows of split partials are then not 16-byte
    aligned, so it stores them one float at a time) against the oracle, and logits written to a
    4-byte-aligned (not 16-byte-aligned) buffer equal the aligned ones bit for bit."""
    from nvfp4_block_scaled_quant_gb300 import _lib
    for E in (21, 24):
        wg, ref = _gate(E, 512, 11)
        x = workloads.activations(6, 512, seed=12, device="cpu")
        ids, w, logits = ops.router(x.to(DEV), wg, 3, want_logits=True)
        _check_router(x, wg, ref, 3)
        T, H = x.shape
        xd = x.to(DEV)
        buf = torch.full((T * E + 4,), float("nan"), dtype=torch.float32, device=DEV)
        ids2 = torch.empty(T, 3, dtype=torch.int32, device=DEV)
        w2 = torch.empty(T, 3, dtype=torch.float32, device=DEV)
        n = int(_lib.lib().nvfp4_router_workspace_bytes(T, E))
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device=DEV)
        _lib.call("nvfp4_router", xd.data_ptr(), T, H, wg.data_ptr(), E, 3, ids2.data_ptr(), w2.data_ptr(),
                  buf.data_ptr() + 4, ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert torch.isnan(buf[0]) and torch.isnan(buf[T * E + 1:]).all()
        assert torch.equal(buf[1:T * E + 1].view(T, E), logits)
        assert torch.equal(ids2, ids) and torch.equal(w2, w)
