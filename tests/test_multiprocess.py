"""The N > 1 path of bench.py on CPU: two gloo ranks agree on the slowest
rank's time and on the whole-job throughput, and the reference arm prints
only on rank 0."""
import os
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 100.0 + 50.0 * rank           # rank 1 is the slow one
        slowest = bench.reduce_max(local_ms, world)
        value = bench.aggregate_tflops(10 ** 12, 4, world, slowest)
        out[rank] = (slowest, value)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = 29500 + os.getpid() % 1000
    with mp.get_context("spawn").Manager() as manager:  # no fork of a process holding OpenMP threads
        out = manager.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    slowest, value = res[0]
    assert slowest == 150.0
    # 2 ranks x 4 steps x 1 TFLOP in 0.15 s
    assert value == pytest.approx(2 * 4 * 1.0 / 0.15)


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "c1"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
