"""The benchmark's multi-rank reduction (bench.reduce_over_ranks) on two gloo
ranks on the CPU: the whole-job time is the slowest rank's, the units are summed
over ranks, and every rank gets the same pair."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r ran (r + 1) * 0.5 s over (r + 1) * 100 query rows
        t, u = bench.reduce_over_ranks(0.5 * (rank + 1), 100.0 * (rank + 1), dist)
        out[rank] = (t, u)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True,
                           start_method="spawn")
        got = dict(out)
    assert got[0] == got[1] == (1.0, 300.0)


def test_reduce_single_process_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(2.5, 40.0, None) == (2.5, 40.0)
    if dist.is_available() and not dist.is_initialized():
        assert bench.reduce_over_ranks(2.5, 40.0, dist) == (2.5, 40.0)


@pytest.mark.parametrize("impl", ["reference"])
def test_reference_arm_only_rank0_prints(impl, tmp_path):
    """Under torchrun the reference arm runs on rank 0 alone; other ranks exit 0
    without work (checked through main()'s rank handling with RANK=1)."""
    import subprocess
    import sys
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", impl, "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
