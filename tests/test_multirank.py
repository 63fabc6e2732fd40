"""The benchmark's multi-rank bookkeeping (weak scaling: every rank runs its
own replica; the step time is the slowest rank's) with two gloo ranks on
the CPU."""

import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = [3.0, 5.0][rank]
    slowest = bench.max_over_ranks(ms, "cpu")
    value = bench.whole_job_tflops(1e12, world, slowest)
    out.put((rank, slowest, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slower rank's 5 ms; the job did 2 TFLOP in 5 ms
    assert [r[1] for r in res] == [5.0, 5.0]
    assert all(abs(r[2] - 400.0) < 1e-9 for r in res)


def test_single_process_needs_no_group():
    import bench

    assert bench.max_over_ranks(7.5, "cpu") == 7.5
    assert abs(bench.whole_job_tflops(2e12, 1, 10.0) - 200.0) < 1e-9


def test_bench_launcher_runs_replicas():
    """`bench.py --gpus 2` (no torchrun environment) starts two ranks with
    RANK / WORLD_SIZE set; rank 0 alone prints the line, with n_gpus 2.  The
    reference arm runs on the CPU, so this needs no GPU."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--workload", "single-256", "--steps", "1", "--warmup", "3", "--ref-seconds", "0.1"],
                         env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1  # only rank 0 prints
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["impl"] == "reference"
