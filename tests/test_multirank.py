"""Multi-process host logic on CPU (gloo, world size 2).

The GEMM path runs as independent replicas, one per GPU, with no collective
on the data path; what spans ranks is the benchmark's bookkeeping: the
slowest rank's step time and the whole-job rate, and the reference arm that
rank 0 alone runs.  Neither needs a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step = [0.0015, 0.0020][rank]  # rank 1 is the slower one
        m = bench.max_over_ranks(step, world, torch.device("cpu"))
        q.put((rank, m, bench.whole_job_tflops(1e12, m, world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, m, v in got:
        assert m == pytest.approx(0.0020)  # every rank sees the slowest step
        assert v == pytest.approx(2 * 1e12 / 0.0020 / 1e12)  # both ranks' work over that time


def test_single_rank_is_identity():
    assert bench.max_over_ranks(0.5, 1, None) == 0.5
    assert bench.whole_job_tflops(2e12, 0.5, 1) == pytest.approx(4.0)


def test_reference_arm_under_torchrun_rank0_only():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3", "--gpus", "2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1  # rank 0 alone prints
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
