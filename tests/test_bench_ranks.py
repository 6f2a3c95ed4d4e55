"""Multi-rank path of bench.py on CPU: two gloo ranks, one replica each.

The timed value must be the slowest rank's and `value` must count the
queries of every rank (weak scaling, no data-path collective)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.max_over_ranks(1.5 + rank, world)          # ms per step on this rank
    q = bench.job_queries_per_s(world, 8, t)
    out[rank] = (t, q)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, start_method="spawn")
    assert out[0] == out[1]
    t, q = out[0]
    assert t == 2.5                                       # the slower rank
    assert q == pytest.approx(2 * 8 / 2.5e-3)
