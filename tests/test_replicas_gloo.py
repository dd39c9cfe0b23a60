"""The multi-GPU path of bench.py (replicas) on CPU: two gloo ranks.

The layer has no exchange step, so N GPUs run N independent replicas; the
only cross-rank logic is the rank environment, the barriers around the timed
region, the slowest rank's time and the whole-job throughput.  These run here
exactly as bench.py calls them, with the gloo backend on CPU.
"""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    w, r, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    dist.barrier()
    # rank r "took" 10 + 5r ms for its share; the job took the slowest one's time
    ms = bench.max_over_ranks(10.0 + 5.0 * r, dist, device="cpu")
    value = bench.job_throughput(1000, w, ms)
    dist.barrier()
    with open(os.path.join(out_dir, "rank%d.txt" % r), "w") as f:
        f.write("%d %d %d %r %r\n" % (w, r, local, ms, value))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_every_rank(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    rows = [open(tmp_path / ("rank%d.txt" % r)).read().split() for r in range(world)]
    for r, (w, rank, local, ms, value) in enumerate(rows):
        assert (int(w), int(rank), int(local)) == (world, r, r)
        assert float(ms) == 15.0                    # the slower rank's 15 ms on both ranks
        assert float(value) == 1000 * world / 0.015   # all ranks' units over that time


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(12.5, None) == 12.5
    assert bench.job_throughput(131072, 1, 56.0) == 131072 / 0.056


def test_gpus_flag_starts_that_many_ranks():
    """bench.py --gpus 2, run directly, starts two ranks under
    torch.distributed.run; rank 0 alone prints the line, with n_gpus 2 (the
    oracle arm, which needs no GPU)."""
    import json
    import subprocess

    env = dict(os.environ)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl",
                          "reference", "--workload", "small", "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, env=env, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [json.loads(l) for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    assert lines[0]["n_gpus"] == 2 and lines[0]["impl"] == "reference"
    assert "bench: rank 0 of 2" in res.stderr and "bench: rank 1 of 2" in res.stderr


def test_gpus_flag_must_match_the_launched_ranks():
    import subprocess

    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "4", "--impl",
                          "reference", "--workload", "small"],
                         capture_output=True, text=True, env=env, timeout=300)
    assert res.returncode != 0
    assert "--gpus 4 but WORLD_SIZE=2" in res.stderr
