"""The replica path of bench.py on CPU: two gloo ranks (no GPU) combine their
timings as the slowest rank's and their tokens as the sum, and the reference
arm prints only on rank 0."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, e2e, tok = bench.combine_ranks(10.0 + rank, 20.0 - rank, 7 * (rank + 1), world, "cpu")
        out[rank] = (ms, e2e, tok)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_combine_as_weak_scaling():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    # every rank sees the slowest rank's times and the total tokens
    assert res[0] == res[1] == (11.0, 20.0, 21.0)


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    assert bench.combine_ranks(3.0, 4.0, 5, 1, "cpu") == (3.0, 4.0, 5.0)
