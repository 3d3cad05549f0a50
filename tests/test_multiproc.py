"""CPU tests of bench.py's multi-rank logic with torch.distributed on gloo (world size 2):
the job time is the slowest rank's, the weak-scaling throughput counts every rank's
work, and the reference arm runs on rank 0 only."""

import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as tdist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    my_ms = 100.0 + 50.0 * rank                 # rank 1 is the slower one
    t = bench.max_over_ranks(my_ms, world)
    tdist.barrier()
    tdist.destroy_process_group()
    q.put((rank, t))


def test_max_over_ranks_gloo():
    world, port = 2, 29517
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(world))
    assert got == {0: 150.0, 1: 150.0}


def test_whole_job_tflops_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_tflops(1e12, 10, 1, 1000.0)
    assert one == pytest.approx(10.0)
    assert bench.whole_job_tflops(1e12, 10, 4, 1000.0) == pytest.approx(40.0)
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_reference_arm_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


@pytest.mark.slow
def test_reference_arm_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
