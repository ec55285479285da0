"""CPU checks of the C-ABI library: it builds, loads, exports every declared
symbol, and rejects bad arguments on the host before touching a device."""

import ctypes

import numpy as np
import pytest

from nvfp4_block_scaled_quant_gb300 import _lib
from nvfp4_block_scaled_quant_gb300 import build as B
from oracle import nvfp4_oracle as O


@pytest.fixture(scope="module")
def L():
    B.build()
    return _lib.lib()


def test_exports_every_declared_symbol(L):
    names = _lib.declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_lib._SIGNATURES), "binding signatures and header disagree"
    assert L.nvfp4_abi_version() == _lib.ABI_VERSION


def test_sf_bytes_matches_layout_definition(L):
    for rows, K in [(0, 64), (1, 64), (127, 128), (128, 256), (200, 512), (300, 7168), (49920, 7168)]:
        assert L.nvfp4_sf_bytes(rows, K) == O.sf_bytes(rows, K)


def test_status_strings(L):
    for s in range(9):
        assert L.nvfp4_status_string(s)
    assert L.nvfp4_status_string(99) == b"unknown status"


def _q(L, *args):
    return L.nvfp4_quantize_act(*args)


def test_quantize_rejects_bad_arguments(L):
    buf = ctypes.create_string_buffer(1 << 16)
    p = ctypes.addressof(buf)
    p16 = (p + 15) & ~15
    cases = [
        ((p16, 4, 100, 128, 0, p16, p16, p16, 0, p16, 4096, None), _lib.ERR_UNSUPPORTED_SHAPE),  # K % 64
        ((p16, -1, 64, 64, 0, p16, p16, p16, 0, p16, 4096, None), _lib.ERR_INVALID_ARG),
        ((p16, 4, 64, 64, 7, p16, p16, p16, 0, p16, 4096, None), _lib.ERR_INVALID_ARG),     # gs_mode
        ((p16, 4, 64, 64, 0, p16, p16, p16, 5, p16, 4096, None), _lib.ERR_INVALID_ARG),     # sf_layout
        ((None, 4, 64, 64, 0, p16, p16, p16, 0, p16, 4096, None), _lib.ERR_INVALID_ARG),
        ((p16, 4, 64, 60, 0, p16, p16, p16, 0, p16, 4096, None), _lib.ERR_MISALIGNED),      # ldx < K
        ((p16 + 2, 4, 64, 64, 0, p16, p16, p16, 0, p16, 4096, None), _lib.ERR_MISALIGNED),  # x alignment
        ((p16, 4, 64, 64, 0, p16, p16, p16, 0, p16, 16, None), _lib.ERR_WORKSPACE),
    ]
    for args, want in cases:
        assert _q(L, *args) == want, (args, L.nvfp4_last_error_string())
        assert L.nvfp4_last_error_string().startswith(b"nvfp4_quantize_act")


def test_linear_and_moe_reject_bad_shapes(L):
    p = 1 << 20  # a fake aligned address: validation fails before it is used
    assert L.nvfp4_linear(p, 4, 64, 100, p, p, p, 0, p, p, p, 1 << 20, None) == _lib.ERR_UNSUPPORTED_SHAPE
    assert L.nvfp4_linear(p, 4, 96, 128, p, p, p, 0, p, p, p, 1 << 20, None) == _lib.ERR_UNSUPPORTED_SHAPE
    assert L.nvfp4_linear(p, 4, 64, 128, p, p, p, 0, p, p, p, 16, None) == _lib.ERR_WORKSPACE
    assert L.nvfp4_gemm(p, p, p, 4, 64, 128, None, p, p, p, None) == _lib.ERR_INVALID_ARG
    assert L.nvfp4_gemm(p, p, p, 4, 64, 136, p, p, p, p, None) == _lib.ERR_UNSUPPORTED_SHAPE   # N % 16
    assert L.nvfp4_grouped_linear(p, 4, 2, 64, 144, p, p, p, 0, p, p, p, 1 << 20, None) == _lib.ERR_UNSUPPORTED_SHAPE
    assert L.nvfp4_moe_workspace_bytes(16, 250, 128, 8, 2, 0) == 0       # H % 128
    assert L.nvfp4_moe_workspace_bytes(16, 256, 100, 8, 2, 0) == 0       # I % 64
    assert L.nvfp4_moe_workspace_bytes(16, 256, 128, 2000, 2, 0) == 0    # E too large
    assert L.nvfp4_moe_workspace_bytes(16, 256, 128, 8, 40, 0) == 0      # topk too large
    assert L.nvfp4_moe_route(p, 4, 2, 0, p, p, p, p, None) == _lib.ERR_INVALID_ARG
    assert L.nvfp4_moe_route(p + 1, 4, 2, 8, p, p, p, p, None) == _lib.ERR_MISALIGNED
    n = L.nvfp4_moe_workspace_bytes(16, 256, 128, 8, 2, 1)
    assert L.nvfp4_moe_dispatch(p, 16, 256, 128, 8, 2, p, 1, 0, p, p, n - 1, None) == _lib.ERR_WORKSPACE
    assert L.nvfp4_moe_dispatch(p, 16, 256, 128, 8, 2, p, 1, 3, p, p, n, None) == _lib.ERR_INVALID_ARG
    assert L.nvfp4_moe_forward(p, 16, 256, 128, 8, 2, p, p, p, p, p, p, p, p, None, None, p, None, None, 0, p, p,
                               p, p, n, None) == _lib.ERR_INVALID_ARG  # sh_w2 without sh_w13
    assert L.nvfp4_debug_wait_timeout(0, None) == _lib.ERR_INVALID_ARG


def test_prepared_weight_sizes_and_partial_tiles(L):
    """Prepared codes are whole 128-row tiles of 128-byte slabs: N % 16 is enough for one group
    (the last tile padded), the grouped layouts and the w13 interleave keep N % 128."""
    assert L.nvfp4_prepared_weight_bytes(1, 256, 256) == 256 * 128
    assert L.nvfp4_prepared_weight_bytes(1, 144, 256) == 256 * 128      # 144 rows -> two tiles
    assert L.nvfp4_prepared_weight_bytes(1, 16, 7168) == 128 * 28 * 128
    assert L.nvfp4_prepared_weight_bytes(3, 128, 320) == 3 * 128 * 2 * 128  # K/2 = 160 bytes -> two slabs
    assert L.nvfp4_prepared_weight_bytes(2, 144, 256) == 0
    assert L.nvfp4_prepared_weight_bytes(1, 100, 256) == 0
    p = 1 << 20
    assert L.nvfp4_prepare_weights(p, p, 1, 144, 256, _lib.PREP_W13_INTERLEAVE, p + 4096, p + 8192,
                                   None) == _lib.ERR_UNSUPPORTED_SHAPE
    assert L.nvfp4_prepare_weights(p, p, 2, 144, 256, _lib.PREP_PLAIN, p + 4096, p + 8192,
                                   None) == _lib.ERR_UNSUPPORTED_SHAPE


def test_valid_call_without_a_gpu_fails_cleanly(L):
    """Arguments that pass validation reach the device query; with no GPU it must fail, not crash."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    buf = ctypes.create_string_buffer(1 << 16)
    p = (ctypes.addressof(buf) + 255) & ~255
    st = L.nvfp4_quantize_act(p, 4, 64, 64, 0, p, p, p, 0, p, 4096, None)
    assert st in (_lib.ERR_CUDA, _lib.ERR_UNSUPPORTED_DEVICE)


@pytest.mark.parametrize("T,H,I,E,k,sh", [(16, 256, 128, 8, 2, 0), (16, 256, 128, 8, 2, 1), (1, 7168, 2048, 384, 8, 1),
                                          (128, 7168, 2048, 384, 8, 1), (4096, 7168, 2048, 384, 8, 1), (0, 256, 64, 4, 1, 1),
                                          (8, 7168, 2048, 384, 8, 1), (32, 256, 64, 4, 8, 1), (33, 256, 64, 4, 8, 0)])
def test_moe_workspace_layout(L, T, H, I, E, k, sh):
    lay = _lib.MoeWsLayout()
    assert L.nvfp4_moe_workspace_layout(T, H, I, E, k, sh, ctypes.byref(lay)) == 0
    fields = ["counts", "offsets", "pad_offsets", "tile_offsets", "sorted_idx", "inv_idx", "dest_rows", "tile_table",
              "amax_partials", "xq",
              "xsf", "hq", "hsf", "y_acc", "total"]
    offs = [getattr(lay, f) for f in fields]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert lay.total == L.nvfp4_moe_workspace_bytes(T, H, I, E, k, sh)
    rc = lay.rows_capacity
    assert rc % 128 == 0
    # the padded segments always fit: sum_e roundup(c_e, 128) <= T*k + 127 * min(E, T*k), plus the shared rows
    assert rc >= T * k + (127 * min(E, T * k)) // 128 * 128 + (((T + 127) // 128) * 128 if sh else 0)
    # one int32x4 entry per m tile; tiles are 32 rows high up to T = 128, and a group of c rows
    # takes ceil(c / 32) <= 4 ceil(c / 128) of them, so rc / 32 entries always suffice
    assert lay.amax_partials - lay.tile_table >= rc // 32 * 16
    R = 32 if T <= 128 else 128
    rng = np.random.default_rng(T * 7 + k)
    for ids in (rng.integers(0, E, (T, k)), np.zeros((T, k), np.int64), np.arange(T * k).reshape(T, k) % E):
        c = np.bincount(ids.reshape(-1), minlength=E)
        if sh:
            c = np.append(c, T)
        assert int(((c + 127) // 128 * 128).sum()) <= rc
        assert int(((c + R - 1) // R).sum()) * 16 <= lay.amax_partials - lay.tile_table
    assert lay.xsf - lay.xq >= rc * H // 2 and lay.hq - lay.xsf >= O.sf_bytes(rc, H)
    assert lay.hsf - lay.hq >= rc * I // 2 and lay.y_acc - lay.hsf >= O.sf_bytes(rc, I)
    assert lay.total - lay.y_acc >= T * H * 4
