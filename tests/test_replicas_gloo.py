"""bench.py's multi-GPU path is replicas only: each rank runs its own batch,
and the only inter-rank operations are a barrier and the max of the timed
region over ranks.  That host logic runs here as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(ws)
    my_ms = 10.0 + 5.0 * rank                      # rank 1 is the slow replica
    total = bench.reduce_max(my_ms, ws)
    out[rank] = (total, bench.replica_value(16, 30, total, ws))
    dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_time():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:       # no fork of this threaded process
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    # whole-job throughput: both ranks' queries over the slowest rank's time
    assert res[0][1] == pytest.approx(2 * 16 * 30 / 0.015)
