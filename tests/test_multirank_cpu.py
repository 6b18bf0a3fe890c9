"""The N > 1 path of bench.py on CPU: every rank runs an independent replica
(the method is single-GPU, there is no exchange step), the step time is the
maximum over ranks, and the reported value is the whole-job aggregate.
Two gloo ranks on 127.0.0.1."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 4.0 + rank  # rank 1 is the slow one
    ms = bench.max_over_ranks(local_ms, dist, "cpu")
    out[rank] = (ms, bench.aggregate_value(6597e9, ms, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_and_aggregate():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        ms, value = res[r]
        assert ms == pytest.approx(5.0)
        assert value == pytest.approx(2 * 6597e9 / 5e-3 / 1e12)


def test_single_process_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.aggregate_value(1e12, 1.0, 1) == pytest.approx(1000.0)
