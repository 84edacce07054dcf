"""The N>1 host logic of bench.py on CPU: two gloo ranks.

Each rank runs its own batch, so the only cross-rank step is the timing
reduction: the job's elapsed time is the slowest rank's, the work done is
the sum over ranks.
"""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        assert bench.rank_info() == (rank, rank, world)
        el, units = bench.reduce_timing(1.0 + rank, 100.0 * (rank + 1))
        out[rank] = (el, units)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_reduce_timing_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    assert out[0] == out[1] == (2.0, 300.0)


def test_reduce_timing_single_process_is_identity():
    import bench
    assert bench.reduce_timing(0.5, 7.0) == (0.5, 7.0)
