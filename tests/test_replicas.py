"""The N>1 bench path on CPU: two gloo ranks stand in for two GPUs.

The path has no exchange step, so N GPUs run N independent replicas. What
ranks share is the timing: each replica's timed span is reduced to the
maximum over ranks (the slowest replica sets the job time), and the job's
rate counts the units of all ranks. Only rank 0 prints the JSON line; for
the reference arm the other ranks return at once without work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, spans, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.slowest_replica_ms(spans[rank], dist, "cpu")
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_slowest_replica_sets_the_job_time():
    spans = [10.0, 12.5]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, spans, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 12.5, 1: 12.5}


def test_local_span_without_a_process_group():
    assert bench.slowest_replica_ms(7.25, None, "cpu") == 7.25


def test_job_throughput_counts_every_replica():
    one = bench.job_throughput(1e12, 1, 2.0)
    assert one == pytest.approx(5e14)
    assert bench.job_throughput(1e12, 2, 2.0) == pytest.approx(2 * one)
    # the slowest replica's longer step lowers the whole job's rate
    assert bench.job_throughput(1e12, 2, 2.5) < 2 * one


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="2", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3", "--cpu-seconds", "1"], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
