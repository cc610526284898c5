"""The multi-GPU mode of bench.py runs independent replicas (the block's
weights are not sharded, so there is no exchange step): its only
cross-rank work is the max-over-ranks step time.  Checked here with two
gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = [2.0, 3.5][rank]
    ms, value = bench.aggregate_replicas(ms_local, 64, world, dist, torch.device("cpu"))
    results[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = _free_port()
        mp.start_processes(_rank_main, args=(2, port, results), nprocs=2, join=True,
                           start_method="spawn")
        res = dict(results)
    assert set(res) == {0, 1}
    for ms, value in res.values():
        assert ms == 3.5
        assert value == pytest.approx(2 * 64 / 3.5e-3)


def test_single_replica_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.aggregate_replicas(1.6, 64, 1)
    assert ms == 1.6 and value == pytest.approx(64 / 1.6e-3)
