"""The N > 1 path of bench.py on CPU: two gloo ranks agree on the max of their timings and
on the weak-scaling throughput (no GPU, no data-path collective)."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.reduce_max([0.1 * (rank + 1), 2.0 - rank, 5.0])
    out[rank] = got + [bench.weak_scaling_value(1e9, world, got[0])]
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        assert out[r][:3] == pytest.approx([0.2, 2.0, 5.0])
        assert out[r][3] == pytest.approx(2 * 1e9 / 0.2 / 1e9)


def test_single_process_reduction_is_identity():
    import bench
    assert bench.reduce_max([1.0, 2.0]) == [1.0, 2.0]
