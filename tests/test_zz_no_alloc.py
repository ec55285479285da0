"""The dense linear that allocates nothing (nvfp4_linear_noalloc) against nvfp4_linear.

Callers such as a plugin inside a host inference engine that owns all device
memory, or a serving loop with a fixed memory budget, cannot allocate or lend
a workspace; the no-allocation variant keeps its scratch in a static device
array instead.  Its output must match the workspace version on every call,
also when consecutive calls reuse the array with different shapes and global
scales.  This file is collected last so a stop-at-first-failure run has
already run every other test.
"""

import pytest
import torch

from nvfp4_block_scaled_quant_gb300 import _lib, model, ops, workloads
from tests.helpers import assert_parity, bf16_to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc(x, dw, N, gs, dynamic):
    M, K = x.shape
    y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    _lib.call("nvfp4_linear_noalloc", x.data_ptr(), M, K, N, dw.w.data_ptr(), dw.sf.data_ptr(), dw.ws2.data_ptr(),
              _lib.GS_DYNAMIC if dynamic else _lib.GS_STATIC, gs.data_ptr(), y.data_ptr(),
              torch.cuda.current_stream().cuda_stream)
    return y


@pytest.mark.parametrize("dynamic", [True, False])
def test_noalloc_linear_matches_workspace_linear_on_consecutive_calls(dynamic):
    # consecutive calls on the shared array: other shapes and contents each time; the M = 8 call
    # (one launch that quantises inside the GEMM, no scratch) sits between two scratch-path calls
    cases = [(128, 7168, 256, 1), (8, 1536, 384, 3), (37, 1536, 384, 2)]
    for M, K, N, seed in cases:
        dw = model.make_dense_weight(N, K, seed=400 + seed, device=DEV)
        x = workloads.activations(M, K, seed=410 + seed, device=DEV, outliers=True)
        gs_ref = None if dynamic else torch.tensor([0.0031 * seed], dtype=torch.float32, device=DEV)
        y_ref, g_ref = ops.linear(x, dw.w, dw.sf, dw.ws2, N, gs=gs_ref)
        gs = torch.empty(1, dtype=torch.float32, device=DEV) if dynamic else gs_ref.clone()
        y = _noalloc(x, dw, N, gs, dynamic)
        torch.cuda.synchronize()
        assert gs.item() == g_ref.item()
        assert_parity(bf16_to_np(y), bf16_to_np(y_ref), what=f"no-alloc linear M={M} K={K} N={N}")
        assert ops.device_error() == (0, 0)


def test_noalloc_linear_rejects_shapes_above_the_static_array():
    K, N = 7168, 128
    dw = model.make_dense_weight(N, K, seed=420, device=DEV)
    M = 2048  # needs ~8 MB of scratch, the array holds 4 MiB
    assert int(_lib.lib().nvfp4_linear_workspace_bytes(M, K)) > _lib.LINEAR_NOALLOC_MAX_BYTES
    x = torch.zeros(M, K, dtype=torch.bfloat16, device=DEV)
    gs = torch.empty(1, dtype=torch.float32, device=DEV)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    st = _lib.lib().nvfp4_linear_noalloc(x.data_ptr(), M, K, N, dw.w.data_ptr(), dw.sf.data_ptr(),
                                         dw.ws2.data_ptr(), _lib.GS_DYNAMIC, gs.data_ptr(), y.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    assert st == _lib.ERR_WORKSPACE
    assert b"static array" in _lib.lib().nvfp4_last_error_string()
