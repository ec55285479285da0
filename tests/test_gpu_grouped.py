"""Fixed-group NVFP4 linear (grouped o-projection) on the GPU against the oracle (identical operands)."""

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_quant_gb300 import model, ops, workloads
from oracle import nvfp4_oracle as O
from tests.helpers import assert_parity, bf16_to_np, unpack

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(M, G, K, N, seed, gs=None):
    x = workloads.activations(M, G * K, seed=seed, device="cpu", outliers=True)
    gw = model.make_grouped_weight(G, N, K, seed=seed + 1, device=DEV)
    y, g = ops.grouped_linear(x.to(DEV), gw.w, gw.sf, gw.ws2, G, N,
                              gs=None if gs is None else torch.tensor([gs], dtype=torch.float32, device=DEV))
    torch.cuda.synchronize()
    xq = O.quantize(x.float().numpy(), gs=gs)
    if gs is None:
        assert g.item() == float(xq.gs)
    wq = [O.quantize(workloads.weight(N, K, (seed + 1) * 1009 + i, DEV).float().cpu().numpy()) for i in range(G)]
    for i in range(G):
        assert gw.ws2[i].item() == float(wq[i].gs)
    ref = O.grouped_linear(xq, [w.codes for w in wq], [w.sf for w in wq], [w.gs for w in wq])
    assert_parity(bf16_to_np(y), ref, what=f"grouped linear M={M} G={G} K={K} N={N}")


@pytest.mark.parametrize("M,G,K,N", [(1, 2, 64, 128), (5, 3, 128, 256), (130, 4, 192, 128), (33, 8, 256, 128),
                                     (257, 2, 512, 384)])
def test_grouped_linear_ragged(M, G, K, N):
    _run(M, G, K, N, seed=M * 31 + G)


@pytest.mark.parametrize("M,G,K,N,gs", [(7, 4, 768, 256, None), (32, 2, 512, 128, None), (3, 2, 320, 384, None),
                                        (1, 8, 4096, 1024, 0.0021), (16, 3, 1024, 640, None)])
def test_grouped_linear_fused_shapes(M, G, K, N, gs):
    """At most 32 tokens: the one-launch path (the GEMM CTAs quantise x themselves, one tile per
    CTA, the K stages round-robin over four MMA issuers).  K = 768 and 320 leave issuers without a
    stage (K = 320 ends in a one-step stage), M = 32 and 16 fill the token columns, N = 640 five
    tiles per group.  Every output against the oracle, dynamic and static gs."""
    _run(M, G, K, N, seed=M * 17 + G * 5 + K, gs=gs)
    assert ops.device_error() == (0, 0)


@pytest.mark.parametrize("M", sorted(workloads.GROUPED_LINEAR))
def test_grouped_linear_oproj_workload(M):
    """8 groups x 4096 inputs -> 1024 outputs each, every output checked."""
    _, G, K, N = workloads.GROUPED_LINEAR[M]
    _run(M, G, K, N, seed=500 + M)


def test_grouped_linear_static_gs_and_single_group_equals_linear():
    _run(17, 3, 256, 128, seed=9, gs=0.0021)
    # G = 1 is the dense linear
    x = workloads.activations(9, 256, seed=10, device=DEV)
    dw = model.make_dense_weight(256, 256, seed=11, device=DEV)
    y1, _ = ops.grouped_linear(x, dw.w, dw.sf, dw.ws2, 1, 256)
    y2, _ = ops.linear(x, dw.w, dw.sf, dw.ws2, 256)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
