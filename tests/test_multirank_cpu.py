"""The N-GPU bench path on CPU: two gloo ranks, each with its own batch, aggregated the way
bench.py reports a multi-GPU run (slowest rank's time, all ranks' retained pairs)."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r pretends its timed region took 10*(r+1) ms and kept 1000*(r+1) pairs
    ms, retained = bench.aggregate_over_ranks(10.0 * (rank + 1), 1000 * (rank + 1), dist, "cpu")
    out[rank] = (ms, retained, bench.pairs_per_second(retained, 5, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_with_gloo():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    for r in range(world):
        ms, retained, pps = out[r]
        assert ms == pytest.approx(20.0)          # the slowest rank sets the time
        assert retained == pytest.approx(3000.0)  # pairs of every rank count
        assert pps == pytest.approx(3000.0 * 5 / 0.020)


def test_single_rank_aggregation_is_identity():
    import bench
    assert bench.aggregate_over_ranks(12.5, 777) == (12.5, 777.0)
    assert bench.pairs_per_second(1000, 10, 5.0) == pytest.approx(2e6)
