"""The N > 1 path of the benchmark (independent replicas) on CPU: two gloo ranks.

Each rank reports its own timed region and units; the job's figure must be all
ranks' units over the slowest rank's time, the same on every rank.
"""

import socket

import pytest
import torch.multiprocessing as mp

from nvfp4_block_scaled_quant_gb300 import replicas


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, times_ms, units, out):
    import os

    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert replicas.env_ranks() == (rank, world, rank)
        dist.barrier()
        out.put((rank, replicas.replica_throughput(times_ms[rank], units[rank])))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times_ms,units", [((100.0, 200.0), (1000.0, 1001.0)), ((50.0, 50.0), (4096.0, 4096.0))])
def test_two_gloo_ranks_aggregate_max_time_and_all_units(times_ms, units):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times_ms, units, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    want_ms = max(times_ms)
    want_units = sum(units)
    for r in range(2):
        value, ms, u = got[r]
        assert ms == want_ms and u == want_units
        assert value == pytest.approx(want_units / (want_ms / 1e3), rel=1e-12)


def test_single_process_is_the_local_figure():
    assert replicas.replica_throughput(250.0, 1000.0) == (4000.0, 250.0, 1000.0)


@pytest.mark.parametrize("gpus,env,want", [
    (1, {}, "run"),
    (8, {}, "relaunch"),
    (2, {"WORLD_SIZE": "2", "RANK": "1"}, "run"),
    (1, {"WORLD_SIZE": "1"}, "run"),
    (8, {"WORLD_SIZE": "4"}, "error"),
    (1, {"WORLD_SIZE": "2"}, "error"),
    (0, {}, "error"),
])
def test_launch_plan_of_the_gpus_flag(gpus, env, want):
    """--gpus N without a launcher starts N local ranks; under a launcher it must agree with
    WORLD_SIZE (a silent one-GPU run for --gpus 8 is an error)."""
    action, why = replicas.launch_plan(gpus, env)
    assert action == want
    assert (why != "") == (want == "error")
