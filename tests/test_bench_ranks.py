"""bench.py's multi-rank path on CPU: N replicas (one per GPU on a GPU machine),
timed as the slowest rank, whole-job ms per linear over all ranks' linears.
Two gloo ranks on 127.0.0.1 stand in for two GPUs; nothing here needs a GPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank)      # rank 1 is the slower replica
        out[rank] = (slowest, bench.job_ms_per_linear(slowest, 3, world))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_and_count_every_rank():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1] == (15.0, 15.0 / 6)


def test_single_process_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_ms_per_linear(9.0, 3, 1) == pytest.approx(3.0)
