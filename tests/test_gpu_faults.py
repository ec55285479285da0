"""Device-side failure detection without a GPU fault.

* A bounded wait on a barrier nothing arrives at gives up after its limit,
  raises the timeout flag and the context stays usable.
* Expert ids outside [0, E) are dropped and flagged; the rest of the MoE
  output is still computed.
"""

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_quant_gb300 import _lib, model, ops, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_bounded_wait_times_out_and_context_survives():
    ops.device_error()
    ops.debug_wait_timeout(20000)  # 20 ms
    st, flags = ops.device_error()
    assert st == _lib.ERR_TIMEOUT and flags & _lib.DEVERR_PIPELINE_TIMEOUT
    assert not flags & 0x80000000, "the barrier reported completion although nothing arrived"
    # the context still works
    x = torch.ones(4, 64, dtype=torch.bfloat16, device=DEV)
    q, sf, gs = ops.quantize_act(x)
    torch.cuda.synchronize()
    assert gs.item() == np.float32(1.0) / np.float32(2688.0)
    assert ops.device_error() == (0, 0)


def test_moe_bad_expert_id_is_flagged():
    T, H, I, E, k = 8, 256, 128, 4, 2
    W = model.make_moe_weights(E, H, I, 107, DEV, shared=False)
    x = workloads.activations(T, H, seed=1, device=DEV)
    ids = torch.tensor([[0, 1]] * T, dtype=torch.int32, device=DEV)
    w = torch.full((T, k), 0.5, device=DEV)
    a2 = torch.full((E + 1,), 0.01, device=DEV)
    y_ok, _ = ops.moe_forward(x, ids, w, W, a2)
    ids_bad = ids.clone()
    ids_bad[3, 1] = 7
    ops.device_error()
    y_bad, _ = ops.moe_forward(x, ids_bad, w, W, a2)
    st, flags = ops.device_error()
    assert st == _lib.ERR_DEVICE_FAULT and flags == _lib.DEVERR_BAD_EXPERT_ID
    diff = (y_ok.float() - y_bad.float()).abs().amax(dim=1)
    assert (diff[torch.arange(T, device=DEV) != 3] == 0).all() and diff[3] > 0
    assert torch.isfinite(y_bad.float()).all()
