"""Host logic of bench.py's multi-rank path, on CPU with gloo (world size 2).

The block does not shard across GPUs here (replicas only): each rank runs an
independent replica, and the reported throughput is the units all ranks
processed divided by the slowest rank's time.  This checks the max/sum
reductions and the aggregation on two CPU ranks, and that a rank that fails
is seen by the other through the process-group timeout rather than a hang.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    bench.dist_init("gloo")
    seconds = [2.0, 3.0][rank]
    units = [10.0, 20.0][rank]
    mx = bench.reduce_max(seconds)
    sm = bench.reduce_sum(units)
    bench.barrier()
    out[rank] = (mx, sm, bench.aggregate_throughput(sm, mx))
    dist.destroy_process_group()


def test_replica_aggregation_two_gloo_ranks():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    for r in range(2):
        mx, sm, thr = out[r]
        assert mx == 3.0 and sm == 30.0 and thr == pytest.approx(10.0)


def _failing_worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    from datetime import timedelta

    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=timedelta(seconds=5))
    if rank == 1:
        os._exit(3)  # leaves between steps, with nothing in flight
    import bench
    try:
        bench.reduce_max(1.0)
        out[rank] = "no error"
    except Exception as e:  # the survivor learns of it through the collective
        out[rank] = type(e).__name__


def test_lost_rank_surfaces_as_error_not_hang():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    ctx = mp.start_processes(_failing_worker, args=(2, port, out), nprocs=2, start_method="spawn",
                             join=False)
    for p in ctx.processes:
        p.join(60)
    assert all(not p.is_alive() for p in ctx.processes)
    assert out.get(0) not in (None, "no error")
