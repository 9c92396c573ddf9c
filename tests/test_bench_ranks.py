"""bench.py's multi-rank path on CPU: N replicas (one per GPU),
timed as the slowest rank, whole-job ms per linear over all ranks' linears.
Two gloo ranks on 127.0.0.1 stand in for two GPUs, each running its own CPU
stand-in of a step through the same timed region the GPU path uses; nothing
here needs a GPU."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import time

    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank)      # rank 1 is the slower replica
        steps = []

        def run():                                              # a replica's timed steps: rank 1 takes longer
            for _ in range(3):
                time.sleep(0.02 * (rank + 1))
                steps.append(rank)

        region = bench.timed_region(run, bench.HostTimer(), world)
        out[rank] = (slowest, bench.job_ms_per_linear(slowest, 3, world), region, len(steps))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_and_count_every_rank():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][:2] == res[1][:2] == (15.0, 15.0 / 6)
    # both ranks report the slower replica's region (3 x 40 ms), and each ran its own 3 steps
    assert res[0][2] == res[1][2]
    assert 115.0 <= res[0][2] < 400.0
    assert res[0][3] == res[1][3] == 3


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_ms_per_linear(9.0, 3, 1) == pytest.approx(3.0)
    t = bench.HostTimer()
    assert bench.timed_region(lambda: None, t, 1) >= 0.0


def test_gpus_must_match_the_launched_ranks():
    sys.path.insert(0, ROOT)
    import bench
    bench.check_world(1, 1)
    bench.check_world(4, 4)
    with pytest.raises(SystemExit, match="nproc-per-node 8"):
        bench.check_world(8, 1)
    # the script itself refuses --gpus 2 without a launcher (before touching a GPU)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "1"],
                       capture_output=True, text=True, env={k: v for k, v in os.environ.items() if k != "WORLD_SIZE"})
    assert r.returncode != 0 and "WORLD_SIZE=1" in r.stderr


def test_digests_are_sha256_of_the_bytes():
    import hashlib

    import torch
    sys.path.insert(0, ROOT)
    import bench
    a = torch.arange(10, dtype=torch.int16)
    b = torch.tensor([1.5], dtype=torch.float32)
    want = hashlib.sha256(a.numpy().tobytes() + b.numpy().tobytes()).hexdigest()
    assert bench.sha256_of([a, b]) == want
    assert bench.digests({"x": [a, b], "y": [b]}) == {"x": want, "y": hashlib.sha256(b.numpy().tobytes()).hexdigest()}
