"""(b) routing on the GPU against the oracle: counts, offsets and both permutations bit-exact."""

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_quant_gb300 import _lib, ops, workloads
from oracle import nvfp4_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check(ids: np.ndarray, E: int):
    c, o, s, inv = ops.moe_route(torch.from_numpy(ids.astype(np.int32)).to(DEV), E)
    torch.cuda.synchronize()
    ref = O.route(ids, E)
    np.testing.assert_array_equal(c.cpu().numpy(), ref.counts)
    np.testing.assert_array_equal(o.cpu().numpy(), ref.offsets)
    np.testing.assert_array_equal(s.cpu().numpy(), ref.sorted_idx)
    np.testing.assert_array_equal(inv.cpu().numpy(), ref.inv_idx)


@pytest.mark.parametrize("cfg", [workloads.TINY, workloads.DECODE[1], workloads.DECODE[8], workloads.DECODE[64],
                                 workloads.PREFILL])
def test_route_workloads(cfg):
    ids, _ = workloads.routing(cfg, seed=99, device="cpu")
    _check(ids.numpy(), cfg.E)


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (3, 2, 5), (100, 4, 7), (33, 32, 1024), (4096, 8, 384)])
def test_route_random_with_duplicates(T, k, E):
    rng = np.random.default_rng(T + k + E)
    _check(rng.integers(0, E, (T, k)), E)


def test_route_skewed_and_empty():
    _check(np.zeros((64, 8), np.int64), 384)           # everything on expert 0
    _check(np.full((5, 2), 383, np.int64), 384)        # last expert only
    c, o, s, inv = ops.moe_route(torch.zeros(0, 8, dtype=torch.int32, device=DEV), 16)
    torch.cuda.synchronize()
    assert c.sum().item() == 0 and o.cpu().tolist() == [0] * 17


def test_route_bad_id_is_flagged_and_dropped():
    ids = np.array([[0, 3], [9, 1], [-2, 2]])
    ops.device_error()  # clear
    c, o, s, inv = ops.moe_route(torch.from_numpy(ids.astype(np.int32)).to(DEV), 4)
    st, flags = ops.device_error()
    assert st == _lib.ERR_DEVICE_FAULT and flags & _lib.DEVERR_BAD_EXPERT_ID
    assert c.cpu().tolist() == [1, 1, 1, 1]
    inv = inv.cpu().numpy()
    assert inv[2] == -1 and inv[4] == -1
    valid = np.array([0, 3, 1, 2])
    ref = O.route(valid.reshape(-1, 1), 4)
    assert c.cpu().tolist() == ref.counts.tolist()
    assert ops.device_error() == (0, 0)
