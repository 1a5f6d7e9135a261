"""bench.py's multi-rank arithmetic on CPU with gloo, world size 2: every
rank reports the slowest rank's time (max over ranks) and the whole-job
time per call divides by steps x ranks.  The data path has no collective;
this is the only cross-rank step (replicas)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_setup(None)
        assert (w, r, local) == (world, rank, rank)
        dist.barrier()
        out[rank] = bench.max_over_ranks(values[rank], w)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    world, port = 2, _free_port()
    values = [12.5, 31.25]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, values, out), nprocs=world, join=True)
        got = dict(out)
    assert got == {0: 31.25, 1: 31.25}


def test_per_call_us_counts_all_replicas():
    # 2 ranks x 10 calls, the slowest rank took 50 ms: 20 calls in 50 ms = 2500 us per call
    assert bench.per_call_us(50.0, 10, 2) == pytest.approx(2500.0)
    assert bench.per_call_us(50.0, 10, 1) == pytest.approx(5000.0)


def test_single_rank_needs_no_process_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(7.0, 1) == 7.0


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun only rank 0 times the oracle and prints the line; any
    other rank exits 0 at once, printing nothing."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       cwd=root, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
