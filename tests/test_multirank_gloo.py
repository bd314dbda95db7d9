"""The N > 1 host path of bench.py on CPU with the gloo backend (world size
2): the step has no cross-GPU exchange, so ranks are independent replicas
and only the timing reduction (slowest rank) crosses ranks; the reference
arm prints on rank 0 only."""

import json
import os
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.5 + rank, world)      # rank 1 is slower
        work = dict(kv_bytes=10 ** 9, tokens=1000)
        value = world * bench.metric_of(work, "GB/s", ms * 1e-3)
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time():
    world, port = 2, 29517
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(world))
    for rank, ms, value in res:
        assert ms == 2.5                      # max over ranks
        assert abs(value - 2 * 1.0 / 2.5e-3) < 1e-6  # both replicas' bytes over the slowest time


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--workload", "tiny"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--workload", "tiny", "--ref-budget", "1"], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
