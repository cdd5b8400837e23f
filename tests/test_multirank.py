"""The N>1 path of bench.py (replicas, one per rank) on CPU with the gloo backend.

Every rank runs its own full workload; only the barrier and the max-over-ranks timing cross
ranks. This checks that timing aggregation and the weak-scaling rate over two ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r pretends its step took (r + 1) seconds and its decode (r + 1) / 2 seconds
    total, dec = bench.max_over_ranks(dist, [rank + 1.0, (rank + 1) / 2.0], "cpu")
    rate = bench.weak_scaling_rate(1000.0, world, total)
    dist.barrier()
    out[rank] = torch.tensor([total, dec, rate], dtype=torch.float64)
    dist.destroy_process_group()


def test_two_rank_timing_is_max_over_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        total, dec, rate = out[r].tolist()
        assert total == 2.0 and dec == 1.0
        assert rate == pytest.approx(1000.0 * 2 / 2.0)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(None, [1.5, 2.5], "cpu") == [1.5, 2.5]
    assert bench.weak_scaling_rate(10.0, 1, 2.0) == 5.0
