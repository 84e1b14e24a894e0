"""The N > 1 host path of bench.py on CPU: gloo ranks, world size 2.

The draft path shards over independent requests with no data-path exchange, so several GPUs run
independent replicas; the only collective is the max over ranks of the step times, and the
whole-job rate counts every rank's units.  These tests run that reduction and the reference
arm's rank handling with gloo processes on the host (no GPU).
"""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # rank r measured (1 + r) ms on the device and (5 - r) ms end to end
        ms, e2e = bench.ranks_max(dist, [1.0 + rank, 5.0 - rank], device="cpu")
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{ms} {e2e} {bench.job_rate(world, 7, ms)}\n")
    finally:
        dist.destroy_process_group()


def test_ranks_max_over_gloo(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for r in range(world):
        ms, e2e, rate = map(float, open(tmp_path / f"rank{r}.txt").read().split())
        assert ms == 2.0 and e2e == 5.0          # the slowest rank's times, on every rank
        assert rate == pytest.approx(2 * 7 / 2e-3)  # both ranks' units over the slowest time


def test_ranks_max_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.ranks_max(None, [3, 4.5]) == [3.0, 4.5]
    assert bench.job_rate(1, 7, 0.5) == pytest.approx(14000.0)


def test_reference_arm_only_rank0_works():
    # under torchrun every rank starts bench.py; the reference arm runs on rank 0 alone
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
