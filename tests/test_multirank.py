"""The N > 1 bench path on CPU: world-size-2 gloo ranks.

The collective path runs as independent replicas, one per GPU, with no data
exchange between ranks; what ranks share is the barrier around the timed
region and the max over ranks of the timed total.  These tests run that
logic with the gloo backend on 127.0.0.1.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        slowest = bench.max_over_ranks(local_ms[rank])
        dist.barrier()
        value = bench.whole_job_gbs(1_000_000_000, 10, world, slowest)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_whole_job_value(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    local_ms = [12.5, 20.0, 7.0, 9.0][:world]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, local_ms, q))
             for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slowest = max(local_ms)
    for rank, got_max, value in out:
        assert got_max == slowest
        # every rank's units over the slowest rank's time
        assert abs(value - world * 1e9 * 10 / (slowest / 1e3) / 1e9) < 1e-9


def test_single_process_is_its_own_max():
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_gbs(2_000_000_000, 4, 1, 1000.0) == 8.0


def test_reference_arm_other_ranks_do_nothing(capsys):
    import types

    import bench

    bench.run_reference(types.SimpleNamespace(workload="allgather_bf16_R8_n8Mi", steps=1,
                                              warmup=0), rank=1, world=2)
    assert capsys.readouterr().out == ""
