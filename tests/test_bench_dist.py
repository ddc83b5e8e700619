"""The bench's multi-process path on CPU: world-size-2 gloo ranks check the
barrier and the max over ranks that the timings go through, and the whole-job
aggregation; the reference arm prints only on rank 0."""
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


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        barrier, dmax = bench.dist_ops(dist, "cpu")
        barrier()
        got = dmax(1.5 + rank)           # each rank's own timing
        barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(world))
    assert res == {0: 2.5, 1: 2.5}     # every rank times with the slowest rank's number


def test_single_process_ops_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    barrier, dmax = bench.dist_ops(None, "cpu")
    barrier()
    assert dmax(3.25) == 3.25


def test_whole_job_value_scales_with_ranks():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_tbps(1, 317460528, 0.1154)
    assert abs(one - 317460528 / 0.1154e-3 / 1e12) < 1e-12
    assert abs(bench.whole_job_tbps(8, 317460528, 0.1154) - 8 * one) < 1e-9


def test_reference_arm_prints_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env["RANK"], env["LOCAL_RANK"] = "0", "0"
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3", "--ref-seconds", "1"], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
