"""bench.py host logic on CPU: byte counts, the replica plumbing under a
2-rank gloo group, and the reference arm's one-line contract under torchrun."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_algorithmic_bytes():
    # per token: QK 40 heads * 512 + 512 + 8 = 21000 B; DSV4 H=64: 132952 B
    assert bench.qk_bytes(1, 32, 8) - 2 * 256 == 21000
    assert bench.dsv4_bytes(1, 64, 1) - 2 * 1024 == 132952
    assert bench.dsv4_bytes(1, 128, 1) - 2 * 1024 == 264024
    assert bench.dsv4_bytes(2, 64, 1) - bench.dsv4_bytes(2, 64, 0) == 584


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    m = bench.max_over_ranks(1.5 + rank, w, torch.device("cpu"))
    q.put((rank, m))
    dist.destroy_process_group()


def test_replicas_max_over_ranks_gloo():
    if torch.cuda.is_available():
        import pytest
        pytest.skip("this check drives the gloo backend; with a GPU the bench uses NCCL")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 2.5), (1, 2.5)]


def test_reference_arm_one_line_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--cpu-sample-tokens", "32"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "GB/s" and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"
