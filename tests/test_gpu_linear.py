"""(e) dense Nvfp4Linear and the GEMM core on the GPU against the oracle (identical operands)."""

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_quant_gb300 import model, ops, workloads
from oracle import nvfp4_oracle as O
from tests.helpers import assert_parity, bf16_to_np, unpack

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _weights(N, K, seed):
    wb = workloads.weight(N, K, seed, "cpu")
    q, sf, ws2 = model.quantize_weight(wb.to(DEV))
    wq = O.quantize(wb.float().numpy())
    # the weight quantisation (the checkpoint format) is bit-exact with the oracle
    assert ws2.item() == float(wq.gs)
    np.testing.assert_array_equal(unpack(q), wq.codes)
    np.testing.assert_array_equal(sf.cpu().numpy().reshape(N, K // 16), wq.sf)
    wp, sfp = ops.prepare_weights(q, sf, N, K)
    return wp, sfp, ws2, wq


@pytest.mark.parametrize("M,K,N", [(1, 64, 128), (5, 128, 256), (130, 256, 384), (257, 1536, 512), (64, 7168, 256),
                                   (128, 128, 128), (100, 512, 256), (300, 192, 640)])
def test_linear_ragged_shapes(M, K, N):
    x = workloads.activations(M, K, seed=M + K + N, device="cpu", outliers=True)
    wp, sfp, ws2, wq = _weights(N, K, seed=M * 7 + N)
    y, gs = ops.linear(x.to(DEV), wp, sfp, ws2, N)
    torch.cuda.synchronize()
    xq = O.quantize(x.float().numpy())
    assert gs.item() == float(xq.gs)
    assert_parity(bf16_to_np(y), O.linear(xq, wq.codes, wq.sf, wq.gs), what=f"linear {M}x{K}x{N}")


@pytest.mark.parametrize("M,K,N", [(1, 256, 16), (5, 512, 144), (32, 128, 400), (3, 4160, 144), (48, 256, 1936),
                                   (130, 1536, 272), (600, 320, 400)])
def test_linear_output_width_multiple_of_16(M, K, N):
    """N % 16 == 0 but not % 128: the prepared weight ends in a partial 128-row tile (zero codes
    and scales from row N on) and only the first N output columns are written.  The fused path
    (M <= 32, small K), the small-A ring (K > 4096), the 128-row tiles (M = 48, 130) and M >= 512,
    where N % 256 != 0 keeps the one-SM tiles; through nvfp4_linear and nvfp4_gemm, every output
    checked, and nothing written past the output."""
    x = workloads.activations(M, K, seed=M + 5 * K + N, device="cpu", outliers=True)
    wp, sfp, ws2, wq = _weights(N, K, seed=M + 3 * N)
    assert wp.numel() == (N + 127) // 128 * 128 * ((K // 2 + 127) // 128) * 128
    xd = x.to(DEV)
    y, gs = ops.linear(xd, wp, sfp, ws2, N)
    q, sf, gq = ops.quantize_act(xd)
    sentinel = torch.full((M * N + 512,), -7.0, dtype=torch.bfloat16, device=DEV)
    y2 = ops.gemm(q, sf, gq, K, wp, sfp, ws2, N, out=sentinel[:M * N].view(M, N))
    torch.cuda.synchronize()
    assert ops.device_error() == (0, 0)
    assert bool((sentinel[M * N:] == -7.0).all())
    xq = O.quantize(x.float().numpy())
    assert gs.item() == float(xq.gs)
    ref = O.linear(xq, wq.codes, wq.sf, wq.gs)
    assert_parity(bf16_to_np(y), ref, what=f"linear {M}x{K}x{N}")
    assert_parity(bf16_to_np(y2), ref, what=f"gemm {M}x{K}x{N}")


@pytest.mark.parametrize("M,K,N", [(512, 256, 256), (700, 320, 512), (640, 1536, 768), (1000, 64, 256),
                                   (1300, 7168, 512), (2049, 512, 1024), (10240, 704, 512)])
def test_linear_pair_tiles_ragged(M, K, N):
    """Shapes of the CTA-pair path (M >= 512, N % 256 == 0, 256 x 256 tiles): M not a multiple
    of 256 (a last tile whose second half starts past the padded scale rows at M = 640 and
    M = 2049), K with a short last stage (K = 320, 64), every output checked, through
    nvfp4_linear and nvfp4_gemm.  M = 10240, N = 512 is 80 tiles, so clusters take two tiles
    in turn; K = 704 is three stages (the last of three K steps), so the two turn-taking MMA
    issuers alternate in opening a tile."""
    x = workloads.activations(M, K, seed=M + 3 * K + N, device="cpu", outliers=True)
    wp, sfp, ws2, wq = _weights(N, K, seed=M + N)
    xd = x.to(DEV)
    y, gs = ops.linear(xd, wp, sfp, ws2, N)
    q, sf, gq = ops.quantize_act(xd)
    y2 = ops.gemm(q, sf, gq, K, wp, sfp, ws2, N)
    torch.cuda.synchronize()
    assert ops.device_error() == (0, 0)
    xq = O.quantize(x.float().numpy())
    assert gs.item() == float(xq.gs)
    ref = O.linear(xq, wq.codes, wq.sf, wq.gs)
    assert_parity(bf16_to_np(y), ref, what=f"pair linear {M}x{K}x{N}")
    assert_parity(bf16_to_np(y2), ref, what=f"pair gemm {M}x{K}x{N}")


@pytest.mark.parametrize("M,K,N", [(10, 1536, 256), (11, 1536, 256), (4, 4096, 384), (1, 4096, 128), (1, 4160, 128),
                                   (2, 64, 1024), (2, 256, 20480), (2, 1536, 19584), (3, 768, 512), (7, 320, 256),
                                   (32, 512, 384)])
def test_linear_fused_quantisation_edges(M, K, N):
    """Small M: the GEMM CTAs quantise x themselves (up to 16K elements, K <= 4096, every K stage
    resident); just beyond those limits the separate quantise launch runs.  Both give the same
    result and the same dynamic gs.  N = 20480 and 19584 have more tiles (160, 153) than SMs, so
    CTAs reuse their resident A for a second tile (one K stage, six K stages).  The K stages go
    round-robin to four MMA issuers, an accumulator each: K = 64, 256, 320 and 768 leave some of them without a stage (K = 320 ends
    in a one-step stage); M = 32 fills every token column of the accumulators."""
    x = workloads.activations(M, K, seed=M * 31 + K, device="cpu", outliers=True)
    wp, sfp, ws2, wq = _weights(N, K, seed=M + N)
    y, gs = ops.linear(x.to(DEV), wp, sfp, ws2, N)
    torch.cuda.synchronize()
    assert ops.device_error() == (0, 0)
    xq = O.quantize(x.float().numpy())
    assert gs.item() == float(xq.gs)
    assert_parity(bf16_to_np(y), O.linear(xq, wq.codes, wq.sf, wq.gs), what=f"linear {M}x{K}x{N}")
    gst = torch.tensor([0.0017], dtype=torch.float32, device=DEV)
    y2, g2 = ops.linear(x.to(DEV), wp, sfp, ws2, N, gs=gst)
    torch.cuda.synchronize()
    assert g2.item() == np.float32(0.0017)  # a static scale is read, not rewritten
    xq2 = O.quantize(x.float().numpy(), gs=np.float32(0.0017))
    assert_parity(bf16_to_np(y2), O.linear(xq2, wq.codes, wq.sf, wq.gs), what=f"linear static {M}x{K}x{N}")


@pytest.mark.parametrize("M", sorted(workloads.DENSE_LINEAR))
def test_linear_dense_workload_full(M):
    """The dense Nvfp4Linear workload (K=1536, N=16384, outlier activations), every output checked."""
    _, K, N = workloads.DENSE_LINEAR[M]
    x = workloads.activations(M, K, seed=20 + M, device="cpu", outliers=True)
    wp, sfp, ws2, wq = _weights(N, K, seed=21)
    y, gs = ops.linear(x.to(DEV), wp, sfp, ws2, N)
    torch.cuda.synchronize()
    xq = O.quantize(x.float().numpy())
    assert gs.item() == float(xq.gs)
    assert_parity(bf16_to_np(y), O.linear(xq, wq.codes, wq.sf, wq.gs), what=f"dense linear M={M}")


def test_linear_static_gs_and_empty():
    M, K, N = 7, 256, 128
    x = workloads.activations(M, K, seed=3, device="cpu")
    wp, sfp, ws2, wq = _weights(N, K, seed=4)
    gs = torch.tensor([0.0021], dtype=torch.float32, device=DEV)
    y, g = ops.linear(x.to(DEV), wp, sfp, ws2, N, gs=gs)
    torch.cuda.synchronize()
    xq = O.quantize(x.float().numpy(), gs=np.float32(0.0021))
    assert_parity(bf16_to_np(y), O.linear(xq, wq.codes, wq.sf, wq.gs), what="static gs")
    y0, _ = ops.linear(torch.empty(0, K, dtype=torch.bfloat16, device=DEV), wp, sfp, ws2, N)
    torch.cuda.synchronize()
    assert y0.shape == (0, N)


@pytest.fixture(scope="module")
def sweep_weight():
    """The 7168 x 7168 weight of the large-GEMM sweep, library- and oracle-side."""
    _, K, N = workloads.DENSE_GEMM[1024]
    return _weights(N, K, seed=31)


def _sweep_rows(M: int, n: int) -> np.ndarray:
    """n seeded rows, always including the first and the last."""
    rows = set(np.random.default_rng(M).choice(M, n - 2, replace=False).tolist()) | {0, M - 1}
    rng = np.random.default_rng(M + 1)
    while len(rows) < n:
        rows.add(int(rng.integers(0, M)))
    return np.array(sorted(rows))


@pytest.mark.parametrize("M,n_rows", [(1024, 48), (4096, 32), (16384, 32)])
def test_gemm_sweep_sampled_rows(sweep_weight, M, n_rows):
    """Large GEMM (K = N = 7168) at the sweep's sizes, in the benchmark's launch configuration:
    the full GPU run through nvfp4_gemm (on quantised activations) and through nvfp4_linear
    (quantisation included); the oracle checks every column of seeded rows.  The global scale
    covers all M rows on both sides."""
    wp, sfp, ws2, wq = sweep_weight
    _, K, N = workloads.DENSE_GEMM[M]
    x = workloads.activations(M, K, seed=30 + M, device="cpu")
    xd = x.to(DEV)
    q, sf, gs = ops.quantize_act(xd)
    y = ops.gemm(q, sf, gs, K, wp, sfp, ws2, N)
    y_lin, gs_lin = ops.linear(xd, wp, sfp, ws2, N)
    torch.cuda.synchronize()
    assert ops.device_error() == (0, 0)
    xf = x.float().numpy()
    g = O.global_scale(xf)
    assert gs.item() == float(g) and gs_lin.item() == float(g)
    rows = _sweep_rows(M, n_rows)
    sub = O.quantize(xf[rows], gs=g)
    ref = O.linear(sub, wq.codes, wq.sf, wq.gs)
    assert_parity(bf16_to_np(y)[rows], ref, what=f"gemm M={M}")
    assert_parity(bf16_to_np(y_lin)[rows], ref, what=f"linear M={M}")
