"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the timing
reduction is a max over ranks, and the reference arm runs on rank 0 only."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(10.0 + 5.0 * rank, dist)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_reference_arm_only_rank0_prints():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--workload", "tiny", "--steps", "1", "--warmup", "0",
                        "--ref-step-seconds", "0.2"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env.update(RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--workload", "tiny", "--steps", "1", "--warmup", "0",
                        "--ref-step-seconds", "0.2"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0
    import json
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def _replica_target(out):
    import bench
    rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
    assert os.environ["LOCAL_RANK"] == str(rank) and os.environ["MASTER_ADDR"] == "127.0.0.1"
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = (world, bench.max_over_ranks(1.0 + rank, dist))
        dist.barrier()
    finally:
        dist.destroy_process_group()
    return 0


def test_run_replicas_sets_the_rank_environment():
    # bench.py --gpus N without a launcher starts N ranks itself; each sees the
    # environment torchrun would set and can rendezvous on 127.0.0.1.
    sys.path.insert(0, ROOT)
    import bench
    out = mp.get_context("spawn").Manager().dict()
    assert bench.run_replicas(3, _replica_target, (out,)) == 0
    assert dict(out) == {0: (3, 3.0), 1: (3, 3.0), 2: (3, 3.0)}


def test_gpus_flag_without_launcher_starts_the_ranks():
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--workload", "tiny", "--steps", "1", "--warmup", "0",
                        "--ref-step-seconds", "0.2"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    import json
    lines = [x for x in r.stdout.strip().splitlines() if x.startswith("{")]
    assert len(lines) == 1  # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2


def _failing_target(out):
    rank = int(os.environ["RANK"])
    if rank == 1:
        raise SystemExit(3)
    dist.init_process_group("gloo", rank=rank, world_size=int(os.environ["WORLD_SIZE"]))
    dist.barrier()  # never completes: rank 1 is gone
    return 0


def test_run_replicas_ends_the_ranks_when_one_fails():
    sys.path.insert(0, ROOT)
    import bench
    import time
    t0 = time.time()
    assert bench.run_replicas(2, _failing_target, (None,)) == 1
    assert time.time() - t0 < 120
