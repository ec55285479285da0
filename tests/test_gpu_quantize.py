"""(a) activation quantisation on the GPU against the oracle: codes, scales and gs bit-exact."""

import ctypes

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_quant_gb300 import _lib, ops, workloads
from oracle import nvfp4_oracle as O
from tests.helpers import unpack, unswizzle

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check(x_bf16: torch.Tensor, gs=None, layout="swizzled"):
    M, K = x_bf16.shape
    q, sf, g = ops.quantize_act(x_bf16.to(DEV), gs=None if gs is None else torch.tensor([gs], device=DEV),
                                sf_layout=layout)
    torch.cuda.synchronize()
    ref = O.quantize(x_bf16.float().numpy(), gs=gs)
    assert g.item() == float(ref.gs) or (np.isnan(g.item()) and np.isnan(ref.gs))
    np.testing.assert_array_equal(unpack(q), ref.codes)
    if layout == "swizzled":
        buf = sf.cpu().numpy()
        np.testing.assert_array_equal(O.unswizzle_sf(buf, M, K), ref.sf)
        # padding rows and columns are written as zero
        full = np.zeros(O.sf_bytes(M, K), dtype=bool)
        full[O.sf_swizzle_offsets(M, K)[:M, : K // 16].ravel()] = True
        assert not buf[~full].any()
    else:
        np.testing.assert_array_equal(sf.cpu().numpy().reshape(M, K // 16), ref.sf)
    return ref


@pytest.mark.parametrize("M,K", [(1, 64), (5, 128), (127, 256), (128, 512), (129, 1536), (300, 7168), (1, 7168),
                                 (16, 256)])
def test_quantize_random_bit_exact(M, K):
    x = workloads.activations(M, K, seed=M * 1000 + K, device="cpu", outliers=K >= 512)
    _check(x)
    _check(x, layout="linear")


def test_quantize_weight_like_and_scaled_inputs():
    for i, scale in enumerate([1e-30, 1e-6, 0.02, 3.0, 1e20, 3e37]):
        x = (workloads.activations(64, 256, seed=i, device="cpu").float() * scale).to(torch.bfloat16)
        _check(x)
    _check(workloads.weight(256, 512, seed=5, device="cpu"), layout="linear")


def test_quantize_static_gs():
    x = workloads.activations(33, 256, seed=7, device="cpu")
    for gs in [0.001, 0.0123, 1.0, 1e-6, 0.0]:  # 1e-6: saturation; 0: all-zero codes
        _check(x, gs=gs)


def test_quantize_rounding_edges():
    """Exact E2M1 midpoints, fp32 neighbours of them, zeros of both signs, saturation."""
    gs = 2.0 ** -7  # block max 6 -> s = 128 exactly, d = 128 * 2^-7 = 1.0, so x * (1/d) == x
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    vals = []
    for m in mids:
        vals += [m, -m]
    vals += [6.0, -0.0, 0.0, 0.1, -0.1, 5.99, 6.0]
    rows = []
    for r in range(0, len(vals), 15):
        blk = vals[r:r + 15]
        blk = blk + [0.0] * (15 - len(blk))
        rows.append([6.0] + blk)  # every block has max 6
    x = np.array(rows, dtype=np.float32).reshape(-1, 16)
    x = np.concatenate([x, np.zeros((x.shape[0], 48), np.float32)], axis=1)
    xb = torch.from_numpy(x).to(torch.bfloat16)  # midpoints and 6 are exact in bf16; 0.1, 5.99 round
    assert xb[0, 1].item() == 0.25 and xb[0, 13].item() == 5.0
    ref = _check(xb, gs=gs)
    assert ref.codes[0, 1] == 0  # 0.25 -> 0 (tie to even)


def test_quantize_zero_rows_and_empty():
    _check(torch.zeros(3, 64, dtype=torch.bfloat16))
    q, sf, g = ops.quantize_act(torch.zeros(0, 64, dtype=torch.bfloat16, device=DEV))
    torch.cuda.synchronize()
    assert g.item() == 0.0 and q.numel() == 0


def test_quantize_strided_rows():
    """ldx > K through the C ABI directly."""
    M, K, ldx = 40, 256, 384
    full = workloads.activations(M, ldx, seed=3, device="cpu")
    xd = full.to(DEV)
    q = torch.empty(M, K // 2, dtype=torch.uint8, device=DEV)
    sf = torch.empty(ops.sf_bytes(M, K), dtype=torch.uint8, device=DEV)
    gs = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(4096, dtype=torch.uint8, device=DEV)
    _lib.call("nvfp4_quantize_act", xd.data_ptr(), M, K, ldx, _lib.GS_DYNAMIC, gs.data_ptr(), q.data_ptr(),
              sf.data_ptr(), _lib.SF_SWIZZLED, ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    ref = O.quantize(full[:, :K].float().numpy())
    assert gs.item() == float(ref.gs)
    np.testing.assert_array_equal(unpack(q), ref.codes)
    np.testing.assert_array_equal(unswizzle(sf, M, K), ref.sf)


def test_prepare_weights_layout():
    """prepare: rows interleaved (64 gate + 64 up per 128) and scales swizzled per group."""
    G, N, K = 3, 256, 192
    rng = np.random.default_rng(0)
    w = rng.integers(0, 256, (G, N, K // 2)).astype(np.uint8)
    sf = rng.integers(0, 127, (G, N, K // 16)).astype(np.uint8)
    for inter in (False, True):
        wo, sfo = ops.prepare_weights(torch.from_numpy(w).to(DEV), torch.from_numpy(sf).to(DEV), N, K,
                                      interleave_w13=inter)
        torch.cuda.synchronize()
        wo, sfo = wo.cpu().numpy(), sfo.cpu().numpy().reshape(G, -1)
        if inter:
            src = np.array([(n // 128) * 64 + (n % 128) if n % 128 < 64 else N // 2 + (n // 128) * 64 + n % 128 - 64
                            for n in range(N)])
        else:
            src = np.arange(N)
        # tile-major codes: block (g, tile, slab) = 128 rows x 128 bytes, the slab past K/2 zero
        slabs = (K // 2 + 127) // 128
        assert wo.size == G * N * slabs * 128
        blocks = wo.reshape(G, N // 128, slabs, 128, 128)
        rows = blocks.transpose(0, 1, 3, 2, 4).reshape(G, N, slabs * 128)
        np.testing.assert_array_equal(rows[:, :, K // 2:], 0)
        for g in range(G):
            np.testing.assert_array_equal(rows[g, :, : K // 2], w[g][src])
            np.testing.assert_array_equal(O.unswizzle_sf(sfo[g], N, K), sf[g][src])
