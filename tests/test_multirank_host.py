"""The N > 1 benchmark path on the CPU (gloo, world size 2): each rank runs
the whole workload (replicas, no collective on the data path); the job time
is the slowest rank's and the value counts every rank's work.  Also the
reference arm's rank handling under a multi-rank launch."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    t = bench.max_over_ranks(1.0 + rank, world, "cpu")          # rank 1 is slower
    v = bench.job_tflops(world, 2e12, 10, t)
    dist.barrier()
    dist.destroy_process_group()
    out[rank] = (t, v)


def test_max_over_ranks_and_job_throughput_gloo():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        t, v = out[r]
        assert t == 2.0                                            # slowest rank
        assert v == pytest.approx(world * 2e12 * 10 / 2.0 / 1e12)  # all ranks' work


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_tflops(1, 1e12, 4, 2.0) == 2.0


def _bench(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], env=env,
                          capture_output=True, text=True, timeout=600, cwd=ROOT)


def test_reference_arm_other_ranks_exit_quietly():
    r = _bench({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--gpus", "2", "--impl",
               "reference",
               "--steps", "1", "--warmup", "1", "--workload", "tiny")
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_json_line():
    r = _bench({"RANK": "0", "WORLD_SIZE": "2", "LOCAL_RANK": "0"}, "--gpus", "2", "--impl",
               "reference", "--steps", "1", "--warmup", "1", "--workload", "tiny",
               "--ref-step-seconds", "1")
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["h2d_bytes_per_step"] == 0


def test_gpus_flag_starts_that_many_ranks():
    """`bench.py --gpus 2` without a launcher starts two ranks itself, so the
    line reports the job's two replicas (reference arm: rank 0 prints)."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                        "--impl", "reference", "--steps", "1", "--warmup", "0",
                        "--workload", "tiny", "--ref-step-seconds", "1"],
                       env=env, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["n_gpus"] == 2 and rec["impl"] == "reference"


def test_gpus_flag_must_match_the_launcher():
    r = _bench({"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"}, "--gpus", "2", "--impl",
               "reference", "--steps", "1", "--warmup", "0", "--workload", "tiny")
    assert r.returncode != 0
    assert "--gpus 2" in r.stderr
