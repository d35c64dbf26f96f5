"""The N>1 path of bench.py on the CPU: two gloo ranks, each with its own
replica's units and time; the job's throughput is the sum of units over the
maximum time.  No GPU, no collective on the data path."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    units, seconds = bench.aggregate(100.0 * (rank + 1), 0.5 + rank, world)
    bench.barrier(world)
    out[rank] = (units, seconds)
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        units, seconds = out[r]
        assert units == pytest.approx(300.0)
        assert seconds == pytest.approx(1.5)


def test_single_rank_is_identity():
    import bench
    assert bench.aggregate(7.0, 2.0, 1) == (7.0, 2.0)
