"""The multi-GPU form of this path is replicas (one independent prompt per rank); the
only cross-rank step is the timing reduction in bench.py. Checked with two gloo ranks on
CPU: every rank gets the slowest rank's time, and barriers pair up."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    ws, r, _ = bench.dist_setup("gloo")
    assert ws == world and r == rank
    bench.barrier(ws)
    m = bench.max_over_ranks(10.0 + 5.0 * rank, ws)
    out[rank] = m
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_max_time():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1] == 15.0
