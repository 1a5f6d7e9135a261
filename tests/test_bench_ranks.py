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


def _bench_env(rank, world):
    return dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                MASTER_ADDR="127.0.0.1", CUDA_VISIBLE_DEVICES="")


@pytest.mark.parametrize("rank", [0, 1])
def test_our_arm_refuses_more_than_one_gpu_before_cuda(rank):
    """Under a torchrun world of two, bench.py's own arm launches nothing: the
    tensor-core kernel's cluster-multicast loads stay on single-GPU calls.
    Rank 0 prints one JSON line with the reason, rank 1 prints nothing, both
    exit 0, and neither imports the library's binding or initialises CUDA
    (the subprocess sees no devices, so any CUDA use would fail)."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    probe = ("import sys, runpy; sys.argv = ['bench.py', '--gpus', '2']; "
             "runpy.run_path('bench.py', run_name='__main__'); "
             "import torch; assert not torch.cuda.is_initialized(); "
             "assert 'speculative_decode_mla_paged_gb300.api' not in sys.modules")
    r = subprocess.run([sys.executable, "-c", probe], cwd=root, env=_bench_env(rank, 2),
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    if rank == 0:
        line = json.loads(r.stdout.strip())
        assert line["n_gpus"] == 2 and "multicast" in line["unavailable"]
    else:
        assert r.stdout.strip() == ""


def test_gpus_flag_alone_is_refused_too():
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "4"], cwd=root,
                       env=_bench_env(0, 1), capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert json.loads(r.stdout.strip())["n_gpus"] == 4
