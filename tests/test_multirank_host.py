"""World-size-2 CPU test of the benchmark's multi-rank host logic (gloo):
every rank times its own replica, the job time is the max over ranks and the
throughput counts the units of all ranks.  No GPU, no data-path collective."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, result):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    my_ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
    t = torch.tensor([my_ms], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    value, tmax = bench.aggregate([float(t.item())] * world, units_per_rank=1.0e9)
    result[rank] = (float(t.item()), value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_over_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    result = mgr.dict()
    mp.start_processes(_worker, args=(world, port, result), nprocs=world, start_method="spawn", join=True)
    assert result[0][0] == result[1][0] == 15.0
    # 2 ranks x 1e9 units over the slowest rank's 15 ms
    assert result[0][1] == pytest.approx(2e9 / 0.015)


def test_aggregate_and_cold_l2_helpers():
    v, t = bench.aggregate([2.0, 4.0, 3.0], 100.0)
    assert t == 4.0 and v == pytest.approx(300.0 / 0.004)
    assert bench.copies_for_cold_l2(42 * 2**20) * 42 * 2**20 >= 4 * bench.L2_BYTES
    assert bench.linear_bytes(20, 6144, 4096) == 6144 * 4096 + 4 * 6144 + 20 * 4096 + 80 + 2 * 20 * 6144
