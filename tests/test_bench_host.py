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
           "--reference-budget-s", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "GB/s" and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"
    # a 1 s budget cannot hold four full steps: a token sample, and the line says so
    S = rec["config"]["tokens_per_step_processed"]
    assert 64 <= S < 32768 and rec["config"]["same_config"] is False
    assert f"first {S} of 32768" in rec["cpu_baseline"]["sample"]


def test_per_config_covers_every_configured_workload():
    """One record per workload the benchmark configurations name: the two
    packed-QKV cases, the two DSV4 cases and the eight sweep points."""
    ws = bench.config_workloads()
    assert [i for i, _, _ in ws] == [0, 1, 2, 3] + [4] * 8
    names = [w.name for _, _, w in ws]
    assert len(set(names)) == len(names) == 12
    sweep = [(w.T, w.H) for i, _, w in ws if i == 4]
    assert sweep == [(1, 128), (17, 128), (1024, 128), (2048, 128), (8192, 128), (32768, 128),
                     (131072, 128), (131072, 64)]


def test_oracle_gbs_on_a_sample():
    """The per-workload CPU figure: the oracle on a token sample, counted by
    the same byte model as the GPU figure."""
    import workloads as wl
    d = wl.make_dsv4(40, 3, max_pos=4096, num_blocks=4, block_size=32, slots="distinct_skip2",
                     seed=5)
    g, S = bench.oracle_gbs("dsv4", d, 16)
    assert S == 16 and g > 0
    d = wl.make_qk(20, 4, 2, 2, max_pos=64, seed=6)
    g, S = bench.oracle_gbs("qk", d, 64)
    assert S == 20 and g > 0


def test_core_bytes_leave_out_tables_indices_and_weights():
    """The narrower byte count differs from the full one by exactly the
    per-token cos/sin rows, positions and slots, and the weight vectors."""
    import workloads as wl
    qk = wl.make_qk(12, 4, 2, 2, max_pos=64, seed=7)
    ds = wl.make_dsv4(10, 3, max_pos=4096, num_blocks=4, block_size=32, slots="distinct_skip2",
                      seed=8)
    b_qk, b_ds = bench.step_bytes(qk, ds)
    tables = 12 * (128 * 4 + 8) + 2 * 128 * 2 + 10 * (64 * 4 + 16) + 2 * 512 * 2
    assert bench.core_bytes(qk, ds) == b_qk + b_ds - tables
    assert bench.core_bytes(qk, ds) == 12 * 6 * 128 * 4 + 10 * (3 * 2048 + 1024) + 8 * 584


def test_one_thread_oracle_baseline():
    import workloads as wl
    qk = wl.make_qk(12, 4, 2, 2, max_pos=64, seed=7)
    ds = wl.make_dsv4(10, 3, max_pos=4096, num_blocks=4, block_size=32, slots="distinct_skip2",
                      seed=8)
    g, S, dt = bench.cpu_baseline_one_thread(qk, ds, *bench.host_step_inputs(qk, ds), tokens=8)
    assert S == 8 and g > 0 and dt > 0
