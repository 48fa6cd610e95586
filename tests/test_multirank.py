"""The multi-process parts of bench.py on CPU: the max-over-ranks reduction with two gloo
ranks, and the reference arm under torchrun with two ranks (rank 0 prints the line, rank 1
exits without work)."""

import json
import os
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        out[rank] = bench.max_over_ranks([1.0 + rank, 5.0 - rank])
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    port = 29500 + (os.getpid() % 1000)
    with mp.get_context("spawn").Manager() as m:  # no fork of a multi-threaded process
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        assert out[0] == [2.0, 5.0] and out[1] == [2.0, 5.0]


def test_max_over_ranks_without_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]


def test_reference_arm_under_torchrun_two_ranks():
    port = 30500 + (os.getpid() % 1000)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--ref-tokens", "1",
           "--workload", "c1_b2_h128_k128"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["cpu_baseline"]["kind"] == "oracle"
    assert d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
