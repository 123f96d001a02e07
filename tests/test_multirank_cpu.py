"""Multi-rank logic of the benchmark on CPU (gloo, world size 2): each rank
runs its own batch of the workload, the step time is the maximum over ranks
and the whole-job value sums the ranks' tokens.  Also runs the reference arm
under torchrun with two ranks: rank 0 alone prints its line."""
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    ms = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
    value = bench.weak_scaling_value(1000, world, ms)
    dist.barrier()
    q.put((rank, ms, value))
    dist.destroy_process_group()


def test_two_rank_aggregation_on_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in out:
        assert ms == 15.0                       # max over ranks
        assert abs(value - 2 * 1000 / 0.015) < 1e-6  # both ranks' tokens over the slowest time


def test_reference_arm_prints_once_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0


@pytest.mark.parametrize("extra", [["--block"], ["--kernel", "gauss"]])
def test_reference_arm_variants(extra):
    # the oracle's variants behind --block and --kernel gauss, one process
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
           "tiny", "--steps", "2", "--warmup", "1"] + extra
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["config"]["block"] == ("--block" in extra)
    assert d["config"]["kernel"] == ("gauss" if "gauss" in extra else "laplace")
