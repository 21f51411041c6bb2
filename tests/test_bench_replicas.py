"""The multi-GPU path of the benchmark is independent replicas (no exchange
step).  Its only cross-rank logic is the aggregation: the job time is the
slowest rank's and the steps of all ranks add up.  Checked with two gloo
ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [100.0, 250.0][rank]          # rank 1 is the slow one
    e2e = [0.5, 0.4][rank]
    res = bench.aggregate(ms, e2e, 10, world, dist, torch.device("cpu"))
    out[rank] = res
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_slowest_rank_and_sums_steps():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn")
    for r in range(world):
        ms, value, e2e_s, e2e_value = out[r]
        assert ms == 250.0 and e2e_s == 0.5
        assert value == pytest.approx(2 * 10 / 0.25)
        assert e2e_value == pytest.approx(2 * 10 / 0.5)


def test_single_rank_aggregation_is_identity():
    import bench
    ms, value, e2e_s, e2e_value = bench.aggregate(64.0, 0.07, 10, 1)
    assert ms == 64.0 and value == pytest.approx(10 / 0.064)
    assert e2e_value == pytest.approx(10 / 0.07)
