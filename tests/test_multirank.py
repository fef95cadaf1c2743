"""The multi-rank host logic of bench.py on CPU (gloo, world size 2): the
timed region's slowest-rank reduction and the weak-scaling aggregate.  Each
rank would drive its own GPU with its own batch; nothing on the data path is
exchanged, so only these two host steps need more than one process."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out[rank] = bench.max_over_ranks(10.0 + 5.0 * rank)   # rank 1 is the slow one
    dist.barrier()
    dist.destroy_process_group()


def test_slowest_rank_time_and_weak_scaling():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()       # no fork of a multi-threaded process
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == 15.0
    import bench
    # two ranks, 1 GB each per step, slowest step 2 ms -> 1000 GB/s whole job
    assert abs(bench.weak_scaling_value(1e9, 2, 2.0) - 1000.0) < 1e-9
    assert bench.max_over_ranks(3.5) == 3.5               # not distributed: identity
