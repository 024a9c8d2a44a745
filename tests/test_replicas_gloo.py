"""bench.py's N > 1 path runs independent replicas (the GEMM has no exchange
step): a barrier, the max of the ranks' times, and a whole-job value of all
ranks' work over that time. Checked here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        t = 1.0 + rank  # rank r "took" 1 + r seconds
        tmax = bench.max_over_ranks(t, world)
        value = bench.aggregate(2 * 64 ** 3, 10, tmax, world)
        out[rank] = (tmax, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.0                     # max over ranks
    want = 2 * 64 ** 3 * 10 * 2 / 2.0 / 1e9                  # both ranks' work / slowest time
    assert res[0][1] == pytest.approx(want) and res[1][1] == pytest.approx(want)


def test_single_rank_is_unchanged():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate(100, 4, 2.0, 1) == pytest.approx(100 * 4 / 2.0 / 1e9)
