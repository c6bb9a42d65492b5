"""The multi-rank bench logic on CPU with two gloo ranks: the timing of a
step is the maximum over ranks, and the job value aggregates every rank's
(replicated) work over that maximum."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [120.0, 180.0][rank]
    ms = bench.reduce_max(local_ms, world, "cpu")
    out[rank] = (ms, bench.aggregate_value(1e12, 10, ms, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        ms, val = out[r]
        assert ms == 180.0
        # 2 ranks x 10 steps x 1 TFLOP in 0.18 s = 111.1 TFLOP/s
        assert val == pytest.approx(2 * 10 * 1e12 / 0.18 / 1e12)


def test_single_rank_identity():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.aggregate_value(2e12, 5, 1000.0, 1) == pytest.approx(10.0)
