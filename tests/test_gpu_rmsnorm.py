"""Fused RMSNorm -> NVFP4 quantisation on the GPU.

A/B (as the fused-vs-unfused harness of page 1): the fused path and the unfused
path (normalise to bf16, then quantise) give bit-identical x_normed, global
scale, codes, scales and GEMM outputs.  Against the oracle: x_normed within one
bf16 unit in the last place of the fp64 RMSNorm; with a static global scale the
codes and scales agree wherever both sides' bf16 x_normed agree, and overall
agreement is >= 99.9 %.
"""

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_quant_gb300 import model, ops, workloads
from oracle import nvfp4_oracle as O
from tests.helpers import assert_parity, bf16_to_np, unpack, unswizzle

pytestmark = pytest.mark.gpu
DEV = "cuda"
EPS = workloads.RMSNORM_EPS


@pytest.mark.parametrize("M,K", [(1, 256), (5, 7168), (128, 7168), (300, 1536)])
@pytest.mark.parametrize("dynamic", [True, False])
def test_fused_equals_unfused(M, K, dynamic):
    x = workloads.activations(M, K, seed=M + K, device=DEV, outliers=True)
    gamma = workloads.norm_weight(K, seed=K, device=DEV)
    gs = None if dynamic else torch.tensor([0.0123], dtype=torch.float32, device=DEV)
    qf, sff, gsf, xn = ops.rmsnorm_quantize(x, gamma, EPS, gs=gs, want_normed=True)
    y = ops.rmsnorm(x, gamma, EPS)
    qu, sfu, gsu = ops.quantize_act(y, gs=None if dynamic else gs.clone())
    torch.cuda.synchronize()
    assert torch.equal(xn, y), "x_normed"
    assert gsf.item() == gsu.item(), "global scale"
    assert torch.equal(qf, qu) and torch.equal(sff, sfu), "codes / scales"
    # GEMM outputs of both paths
    dw = model.make_dense_weight(256, K, seed=7, device=DEV)
    yf = ops.gemm(qf, sff, gsf, K, dw.w, dw.sf, dw.ws2, 256)
    yu = ops.gemm(qu, sfu, gsu, K, dw.w, dw.sf, dw.ws2, 256)
    torch.cuda.synchronize()
    assert torch.equal(yf, yu), "GEMM outputs"


@pytest.mark.parametrize("M,K", [(7, 256), (64, 7168), (130, 1536)])
def test_rmsnorm_quantize_against_oracle(M, K):
    x = workloads.activations(M, K, seed=2 * M + K, device="cpu", outliers=True)
    gamma = workloads.norm_weight(K, seed=K + 1, device="cpu")
    yb, y64, _ = O.rmsnorm(x.float().numpy(), gamma.float().numpy(), EPS)
    # x_normed: within one bf16 ulp of the fp64 value
    xn = bf16_to_np(ops.rmsnorm(x.to(DEV), gamma.to(DEV), EPS))
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(y64), 1e-30))) - 7)
    assert np.all(np.abs(xn - y64) <= ulp * 1.0001)
    same = xn == yb
    assert same.mean() > 0.999
    # codes and scales with a static global scale
    gs = np.float32(np.abs(yb).max() / 2688.0)
    q, sf, _, _ = ops.rmsnorm_quantize(x.to(DEV), gamma.to(DEV), EPS, gs=torch.tensor([gs], device=DEV))
    torch.cuda.synchronize()
    ref = O.quantize(yb, gs=gs)
    codes, sfs = unpack(q), unswizzle(sf, M, K)
    blk_same = same.reshape(M, K // 16, 16).all(axis=2)
    np.testing.assert_array_equal(sfs[blk_same], ref.sf[blk_same])
    np.testing.assert_array_equal(codes.reshape(M, K // 16, 16)[blk_same], ref.codes.reshape(M, K // 16, 16)[blk_same])
    assert (codes == ref.codes).mean() >= 0.999 and (sfs == ref.sf).mean() >= 0.999
    # dynamic global scale: amax / 2688 of the normalised rows
    _, _, g, _ = ops.rmsnorm_quantize(x.to(DEV), gamma.to(DEV), EPS)
    assert g.item() == float(O.global_scale(xn))


def test_rmsnorm_quantize_feeds_linear_within_bound():
    """Normalised, quantised activations through the GEMM against the oracle on identical operands."""
    M, K, N = 32, 1536, 512
    x = workloads.activations(M, K, seed=5, device="cpu", outliers=True)
    gamma = workloads.norm_weight(K, seed=6, device="cpu")
    q, sf, gs, xn = ops.rmsnorm_quantize(x.to(DEV), gamma.to(DEV), EPS, want_normed=True)
    dw = model.make_dense_weight(N, K, seed=8, device=DEV)
    y = ops.gemm(q, sf, gs, K, dw.w, dw.sf, dw.ws2, N)
    torch.cuda.synchronize()
    yb, _, _ = O.rmsnorm(x.float().numpy(), gamma.float().numpy(), EPS)
    xq = O.quantize(yb)
    wq = O.quantize(workloads.weight(N, K, 8, DEV).float().cpu().numpy())
    if np.array_equal(unpack(q), xq.codes) and gs.item() == float(xq.gs):
        assert_parity(bf16_to_np(y), O.linear(xq, wq.codes, wq.sf, wq.gs), what="rmsnorm -> quant -> linear")
    else:  # a bf16 tie in x_normed moved a code: compare at the GEMM's own bound on a looser cosine
        assert O.cosine(bf16_to_np(y), O.linear(xq, wq.codes, wq.sf, wq.gs)) > 0.9999
