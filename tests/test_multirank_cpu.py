"""The benchmark's multi-rank host logic on CPU: two gloo ranks, no GPU.

Under torchrun each rank runs its own replica of the workload; the job rate is
all ranks' steps over the slowest rank's time, and only rank 0 prints.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        local_ms = [120.0, 150.0][rank]
        slowest = bench.max_over_ranks(local_ms)
        rate = bench.job_rate(world, 10, slowest)
        # the reference arm: only rank 0 does work and prints
        buf = io.StringIO()
        args = type("A", (), dict(workload=4, steps=1, warmup=0, gpus=world))()
        with redirect_stdout(buf):
            if rank != 0:
                bench.run_reference(args)
        q.put((rank, slowest, rate, buf.getvalue()))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, rate, printed in out:
        assert slowest == 150.0                      # max over ranks
        assert rate == pytest.approx(2 * 10 / 0.150)  # whole-job steps over the slowest time
        assert printed == ""                         # a non-zero rank of the reference arm prints nothing


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_rate(1, 100, 250.0) == pytest.approx(400.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    """Under torchrun rank 0 alone times the oracle (with the host's cores, not the one BLAS
    thread torchrun gives each rank), prints one JSON line, and every rank exits 0."""
    import json
    import subprocess
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    try:
        host = len(os.sched_getaffinity(0))
    except AttributeError:
        host = os.cpu_count()
    assert d["cpu_baseline"]["cores"] == host
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
