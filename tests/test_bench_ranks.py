"""The multi-process bench logic on the CPU: world size 2 over gloo (no GPU).

Each rank reports its own step time; the job's time is the slowest rank's
(max over ranks) and its throughput counts every rank's tokens."""
import os
import socket
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = textwrap.dedent("""
    import os, sys
    sys.path.insert(0, os.environ["BENCH_ROOT"])
    import torch
    import torch.distributed as dist
    import bench
    ws, rank, local = bench.dist_info()
    dist.init_process_group("gloo")
    mine = [12.5, 30.25][rank]
    got = bench.max_over_ranks(mine, dist, torch.device("cpu"))
    assert got == 30.25, got
    v = bench.job_tokens_per_s(ws, 8192, 30, got)
    assert abs(v - 2 * 8192 * 30 / 0.03025) < 1e-6 * v, v
    dist.barrier()
    dist.destroy_process_group()
    print("rank", rank, "ok")
""")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_dist_info_reads_the_launcher_environment(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "4")
    monkeypatch.setenv("RANK", "3")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.dist_info() == (4, 3, 1)
    assert bench.max_over_ranks(7.0, None, None) == 7.0
    assert bench.job_tokens_per_s(1, 1, 1000, 1000.0) == pytest.approx(1000.0)


def test_two_ranks_take_the_slowest_time():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                   LOCAL_RANK=str(rank), WORLD_SIZE="2", BENCH_ROOT=ROOT, CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", _CHILD], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True))
    outs = []
    for p in procs:
        out, _ = p.communicate(timeout=120)
        outs.append(out)
        assert p.returncode == 0, out
    assert "rank 0 ok" in outs[0] and "rank 1 ok" in outs[1], outs


def test_reference_arm_runs_on_rank_zero_only():
    """Under a launcher with two ranks, rank 1 of the reference arm exits 0
    without work or output (rank 0 alone times the oracle and prints)."""
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "", r.stdout
