"""The multi-process side of bench.py, on CPU: replicas only (every rank runs the
whole block on its own batch, no collective on the data path), so what crosses
ranks is the timing -- the job takes as long as its slowest rank -- and the
reference arm runs on rank 0 alone.  Two gloo ranks stand in for two GPUs."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench
        mine = [12.5, 17.25, 3.0][rank]
        out[rank] = bench.max_over_ranks(mine, world, torch.device("cpu"))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_timing_is_the_slowest_rank_gloo_world2():
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(2, _free_port(), out), nprocs=2, join=True)
        assert dict(out) == {0: 17.25, 1: 17.25}


def test_timing_is_the_slowest_rank_gloo_world3():
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(3, _free_port(), out), nprocs=3, join=True)
        assert dict(out) == {0: 17.25, 1: 17.25, 2: 17.25}


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.5, 1, torch.device("cpu")) == 4.5


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
