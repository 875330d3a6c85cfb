#!/usr/bin/env python
"""Benchmark of the attention-prologue hot path on GB300 (one JSON line).

One step = one pass of the whole hot path over one batch of synthetic input:
  1. fused_qk_norm_rope on packed bf16 QKV [32768, (32+8+8)*128], theta 1e6,
     positions uniform in [0, 131072) -- Q and K normalised and rotated in
     place, V untouched;
  2. dsv4_qnorm_rope_kv_rope_quant_insert on q bf16 [32768, 64, 512] and kv
     [32768, 512], positions uniform in [0, 131072), 65536-slot paged cache,
     slot_mapping a random permutation prefix.
The metric is achieved HBM bandwidth: algorithmic bytes of the step (every
byte the operators must read or write once) / device time of the step, in
GB/s.  Inputs are resident in HBM and larger than L2 (129 MB), so no L2 flush
is needed between steps.

The line also carries:
  * config.core_gbs: the step's rate counted without the cos/sin rows,
    positions, slots and weights (a narrower byte count beside the full one);
  * cpu_baseline.one_thread: the oracle on one host thread, on a token sample;
  * per_config: every workload the benchmark configurations name (the
    17-token and 32768-token packed-QKV cases, the 16-token and 32768-token
    DSV4 cases and each point of the DSV4 token sweep), each under the
    automatic launch shape: median kernel time, GB/s, % of the measured copy
    peak, the time of a plain device copy moving the same bytes (the copy
    ceiling at that launch length), and the CPU oracle's GB/s on a token
    sample of the same workload;
  * context.unfused_torch: the same two operators of the step as separate
    eager PyTorch passes on this GPU (RMSNorm, RoPE, and for DSV4 the
    blockwise scale/cast and the cache scatter), timed and counted with the
    same algorithmic bytes -- what the fusion saves, not a target.
--impl reference times the CPU oracle (the only other implementation of this
path available here) on the same workload (a token sample only when the
requested step count would not finish within about a minute).
--sweep additionally writes per-configuration lines (every workload of the
parity tests, both launch shapes, the dispatch crossover and a 512 MiB
device-to-device copy ceiling) to stderr.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "achieved HBM GB/s and % of GB300 peak, fused norm+RoPE(+quant+insert)"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
PROFILES = os.path.join(ROOT, "profiles")

# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------

def qk_bytes(T, Hq, Hk, D=128, rot=None):
    """Q and K heads read and written once (bf16), one cos/sin row of `rot`
    floats and one position (int64) per token, the two weight vectors once."""
    rot = D if rot is None else rot
    return T * ((Hq + Hk) * D * 2 * 2 + rot * 4 + 8) + 2 * D * 2


def dsv4_bytes(T, H, mapped):
    """q read + written (bf16), kv read (bf16), one 64-float cos/sin row,
    position and slot (int64) per token; 584 bytes per mapped token written;
    the two weight vectors once."""
    return T * (H * 512 * 2 * 2 + 512 * 2 + 64 * 4 + 8 + 8) + mapped * 584 + 2 * 512 * 2


def core_bytes(qk, ds):
    """The step's bytes without the per-token cos/sin rows, positions, slots
    and the weights: Q/K rows read + written, q rows read + written, kv
    vectors read, entries written (the pages define no byte count of their
    own, so this narrower one is reported beside the full one)."""
    T, Hq, Hk, D = qk["qkv"].shape[0], qk["Hq"], qk["Hk"], qk["D"]
    Tq, H = ds["q"].shape[0], ds["H"]
    mapped = int((ds["slot_mapping"] >= 0).sum())
    return T * (Hq + Hk) * D * 4 + Tq * (H * 512 * 4 + 1024) + mapped * 584


def step_bytes(qk, ds):
    return (qk_bytes(qk["qkv"].shape[0], qk["Hq"], qk["Hk"], qk["D"]),
            dsv4_bytes(ds["q"].shape[0], ds["H"], int((ds["slot_mapping"] >= 0).sum())))


def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001
        return FALLBACK_HBM_GBS, "fallback"


DSV4_KERNEL_SOURCES = ("kvq_dsv4.cu", "kvq_device.cuh", "kvq_launch.h")


def kernel_source_hash(files=DSV4_KERNEL_SOURCES):
    """Hash of the sources one kernel is built from (default: the DSV4 kernel)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kv_quant_cache_gb300", "csrc")
    for f in sorted(files):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_tag):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (profiles/*.md carry 'source-hash: <h>' and
    'traffic-bytes-per-launch: <n>' lines)."""
    want = kernel_source_hash()
    if not os.path.isdir(PROFILES):
        return None
    for f in sorted(os.listdir(PROFILES)):
        if not f.startswith(kernel_tag):
            continue
        text = open(os.path.join(PROFILES, f)).read()
        m_h = re.search(r"source-hash:\s*([0-9a-f]+)", text)
        m_t = re.search(r"traffic-bytes-per-launch:\s*([0-9.eE+]+)", text)
        if m_h and m_t and m_h.group(1) == want:
            return float(m_t.group(1))
    return None


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only: no data exchange)
# ---------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def make_step_inputs(device):
    qk = wl.make_qk_workload(wl.QK_LARGE, device=device)
    ds = wl.make_dsv4_workload(wl.DSV4_LARGE, device=device)
    return qk, ds


def launch_qk(kvq, qk, stream):
    kvq.fused_qk_norm_rope(qk["qkv"], qk["Hq"], qk["Hk"], qk["Hv"], qk["D"], qk["eps"],
                           qk["q_weight"], qk["k_weight"], qk["cos_sin"], True, qk["positions"],
                           stream=stream)


def launch_dsv4(kvq, ds, stream):
    kvq.dsv4_qnorm_rope_kv_rope_quant_insert(ds["q"], ds["kv"], ds["eps"], ds["q_weight"],
                                             ds["kv_weight"], ds["cos_sin"], ds["positions"],
                                             ds["slot_mapping"], ds["kv_cache"], stream=stream)


def time_device(kvq, qk, ds, steps, warmup, world, device):
    """Two passes of `steps` steps on one stream.  The timed region proper
    (the step time) has nothing between the launches: consecutive kernels
    overlap their launch with the previous kernel's tail (programmatic
    dependent launch), as in any pipeline.  A second pass records an event
    around every launch for the per-kernel durations; those events cost the
    overlap (about 10 us per step), so that pass gives the kernels' times,
    not the step's."""
    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize(device)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            launch_qk(kvq, qk, stream)
            launch_dsv4(kvq, ds, stream)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    stream.synchronize()
    barrier(world)
    torch.cuda.synchronize(device)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            launch_qk(kvq, qk, stream)
            launch_dsv4(kvq, ds, stream)
        end.record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    total_ms = start.elapsed_time(end)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for e0, e1, e2 in ev:
            e0.record(stream)
            launch_qk(kvq, qk, stream)
            e1.record(stream)
            launch_dsv4(kvq, ds, stream)
            e2.record(stream)
    torch.cuda.synchronize(device)
    qk_ms = [a.elapsed_time(b) for a, b, _ in ev]
    ds_ms = [b.elapsed_time(c) for _, b, c in ev]
    return total_ms, qk_ms, ds_ms


def time_e2e(kvq, qk, ds, steps, device, chunks=8):
    """Same step with host buffers: pinned inputs copied in, the kernels, the
    results (qkv, q, cache) copied out, every step inside the timed region.
    Tokens are independent, so the step is cut into `chunks` token ranges and
    three streams overlap the host->device copy of chunk i+1, the two kernels
    on chunk i and the device->host copy of chunk i-1; consecutive steps hand
    over chunk by chunk, so one step's copies in overlap the previous step's
    copies out (measured 292 -> 318-322 GB/s against a whole-step barrier)."""
    h = {"qkv": qk["qkv"].cpu().pin_memory(), "qk_pos": qk["positions"].cpu().pin_memory(),
         "q": ds["q"].cpu().pin_memory(), "kv": ds["kv"].cpu().pin_memory(),
         "ds_pos": ds["positions"].cpu().pin_memory(),
         "slot": ds["slot_mapping"].cpu().pin_memory()}
    out = {"qkv": torch.empty_like(h["qkv"]).pin_memory(), "q": torch.empty_like(h["q"]).pin_memory(),
           "cache": torch.empty(ds["kv_cache"].shape, dtype=torch.uint8).pin_memory()}
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = sum(t.numel() * t.element_size() for t in out.values())
    T = qk["qkv"].shape[0]
    bounds = [(i * T // chunks, (i + 1) * T // chunks) for i in range(chunks)]
    s_in, s_run, s_out = (torch.cuda.Stream(device) for _ in range(3))
    # per-chunk hand-offs between consecutive steps: chunk i's next inputs
    # wait only for chunk i's results to be out, so the next step's copies in
    # overlap this step's copies out; the next step's first cache writes wait
    # for this step's cache copy
    prev_out = [None] * chunks
    prev_cache = [None]

    def one():
        outs = []
        for i, (a, b) in enumerate(bounds):
            with torch.cuda.stream(s_in):
                if prev_out[i] is not None:
                    s_in.wait_event(prev_out[i])
                qk["qkv"][a:b].copy_(h["qkv"][a:b], non_blocking=True)
                qk["positions"][a:b].copy_(h["qk_pos"][a:b], non_blocking=True)
                ds["q"][a:b].copy_(h["q"][a:b], non_blocking=True)
                ds["kv"][a:b].copy_(h["kv"][a:b], non_blocking=True)
                ds["positions"][a:b].copy_(h["ds_pos"][a:b], non_blocking=True)
                ds["slot_mapping"][a:b].copy_(h["slot"][a:b], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            s_run.wait_event(ev_in)
            if i == 0 and prev_cache[0] is not None:
                s_run.wait_event(prev_cache[0])
            kvq.fused_qk_norm_rope(qk["qkv"][a:b], qk["Hq"], qk["Hk"], qk["Hv"], qk["D"], qk["eps"],
                                   qk["q_weight"], qk["k_weight"], qk["cos_sin"], True,
                                   qk["positions"][a:b], stream=s_run)
            kvq.dsv4_qnorm_rope_kv_rope_quant_insert(
                ds["q"][a:b], ds["kv"][a:b], ds["eps"], ds["q_weight"], ds["kv_weight"],
                ds["cos_sin"], ds["positions"][a:b], ds["slot_mapping"][a:b], ds["kv_cache"],
                stream=s_run)
            ev = torch.cuda.Event()
            ev.record(s_run)
            s_out.wait_event(ev)
            with torch.cuda.stream(s_out):
                out["qkv"][a:b].copy_(qk["qkv"][a:b], non_blocking=True)
                out["q"][a:b].copy_(ds["q"][a:b], non_blocking=True)
                ev_out = torch.cuda.Event()
                ev_out.record(s_out)
            outs.append(ev_out)
        with torch.cuda.stream(s_out):
            out["cache"].copy_(ds["kv_cache"], non_blocking=True)
            ev_cache = torch.cuda.Event()
            ev_cache.record(s_out)
        prev_out[:] = outs
        prev_cache[0] = ev_cache

    one()
    torch.cuda.synchronize(device)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for _ in range(steps):
        one()
    end.record(s_out)
    torch.cuda.synchronize(device)
    return start.elapsed_time(end) / steps, h2d, d2h, chunks


def time_e2e_zero_copy(kvq, qk, ds, steps, device):
    """The step through the C ABI with HOST buffers: the activations and
    indices live in pinned host memory and the kernels read and write them in
    place over NVLink-C2C (weights and tables stay in HBM).  The paged cache
    lives in HBM, where attention reads it; every step also copies the whole
    cache back to pinned host memory (on a second stream, overlapping the next
    step's QK launch), so the step's written entries reach the host inside
    the timed region.  Returns (ms per step, bytes read from host, bytes
    written to host)."""
    hq = {k: v for k, v in qk.items()}
    hd = {k: v for k, v in ds.items()}
    for k in ("qkv", "positions"):
        hq[k] = qk[k].cpu().pin_memory()
    for k in ("q", "kv", "positions", "slot_mapping"):
        hd[k] = ds[k].cpu().pin_memory()
    cache_host = torch.empty(ds["kv_cache"].shape, dtype=torch.uint8).pin_memory()
    stream = torch.cuda.current_stream(device)
    side = torch.cuda.Stream(device)
    T = qk["qkv"].shape[0]
    qk_rows = T * (qk["Hq"] + qk["Hk"]) * qk["D"] * 2          # Q and K heads only
    h2d = (qk_rows + T * 8 + hd["q"].numel() * 2 + hd["kv"].numel() * 2 + T * 8 * 2)
    d2h = qk_rows + hd["q"].numel() * 2 + cache_host.numel()

    def one():
        launch_qk(kvq, hq, stream)
        stream.wait_stream(side)   # the previous step's cache copy is done before this insert
        launch_dsv4(kvq, hd, stream)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            cache_host.copy_(ds["kv_cache"], non_blocking=True)

    one()
    torch.cuda.synchronize(device)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        one()
    stream.wait_stream(side)
    end.record(stream)
    torch.cuda.synchronize(device)
    return start.elapsed_time(end) / steps, h2d, d2h


def host_step_inputs(qk, ds):
    """Host copies of the step's inputs (bf16 as uint16 bits) for the oracle."""
    def h(t):
        return wl.bf16_bits(t) if t.dtype == torch.bfloat16 else wl.host(t)
    return ({k: h(v) for k, v in qk.items() if isinstance(v, torch.Tensor)},
            {k: h(v) for k, v in ds.items() if isinstance(v, torch.Tensor)})


def cpu_baseline(qk, ds, qk_h, ds_h):
    """The oracle as it stands, all host cores, on the whole step's inputs
    (both operators, all 32768 tokens).  Returns (GB/s by the same byte
    count, threads, seconds)."""
    import oracle
    cache = ds_h["kv_cache"].copy()
    t0 = time.perf_counter()
    oracle.qk_norm_rope(qk_h["qkv"], qk["Hq"], qk["Hk"], qk["Hv"], qk["D"], qk["eps"],
                        qk_h["q_weight"], qk_h["k_weight"], qk_h["cos_sin"], qk_h["positions"])
    oracle.dsv4(ds_h["q"], ds_h["kv"], ds["eps"], ds_h["q_weight"], ds_h["kv_weight"],
                ds_h["cos_sin"], ds_h["positions"], ds_h["slot_mapping"], cache)
    dt = time.perf_counter() - t0
    b_qk, b_ds = step_bytes(qk, ds)
    return (b_qk + b_ds) / dt / 1e9, oracle.default_threads(), dt


def cpu_baseline_one_thread(qk, ds, qk_h, ds_h, tokens=1024):
    """The oracle on one host thread, on the first `tokens` tokens of each
    operator.  Returns (GB/s by the same byte model, tokens, seconds)."""
    import oracle
    S = min(tokens, qk_h["qkv"].shape[0], ds_h["q"].shape[0])
    cache = ds_h["kv_cache"].copy()
    t0 = time.perf_counter()
    oracle.qk_norm_rope(qk_h["qkv"][:S], qk["Hq"], qk["Hk"], qk["Hv"], qk["D"], qk["eps"],
                        qk_h["q_weight"], qk_h["k_weight"], qk_h["cos_sin"],
                        qk_h["positions"][:S], nthreads=1)
    oracle.dsv4(ds_h["q"][:S], ds_h["kv"][:S], ds["eps"], ds_h["q_weight"], ds_h["kv_weight"],
                ds_h["cos_sin"], ds_h["positions"][:S], ds_h["slot_mapping"][:S], cache,
                nthreads=1)
    dt = time.perf_counter() - t0
    nb = (qk_bytes(S, qk["Hq"], qk["Hk"], qk["D"])
          + dsv4_bytes(S, ds["H"], int((ds_h["slot_mapping"][:S] >= 0).sum())))
    return nb / dt / 1e9, S, dt


# ---------------------------------------------------------------------------
# context: the unfused PyTorch baseline (separate eager passes on the GPU)
# ---------------------------------------------------------------------------

def unfused_qk(qk):
    """fused_qk_norm_rope as separate eager PyTorch passes (a comparison
    baseline, not part of the library): RMSNorm of the Q heads, RMSNorm of
    the K heads (fp32 results), then NeoX RoPE of each, written back in place
    as bf16.  Intermediates stay fp32 so the result keeps the operator's
    single rounding."""
    T, Hq, Hk, Hv, D = qk["qkv"].shape[0], qk["Hq"], qk["Hk"], qk["Hv"], qk["D"]
    x = qk["qkv"].view(T, Hq + Hk + Hv, D)
    cs = qk["cos_sin"].index_select(0, qk["positions"])
    c, s = cs[:, None, :D // 2], cs[:, None, D // 2:]

    def norm(rows, w):
        return torch.nn.functional.rms_norm(rows.float(), (D,), w.float(), qk["eps"])

    def rope(n):
        a, b = n[..., :D // 2], n[..., D // 2:]
        return torch.cat([a * c - b * s, b * c + a * s], -1)

    nq = norm(x[:, :Hq], qk["q_weight"])
    nk = norm(x[:, Hq:Hq + Hk], qk["k_weight"])
    x[:, :Hq] = rope(nq).to(torch.bfloat16)
    x[:, Hq:Hq + Hk] = rope(nk).to(torch.bfloat16)


def unfused_dsv4(ds):
    """dsv4_qnorm_rope_kv_rope_quant_insert as separate eager PyTorch passes
    (a comparison baseline, not part of the library): RMSNorm + interleaved
    RoPE of q (written back in place) and of kv, the blockwise UE8M0 exponent
    (the smallest e with 448 * 2^e >= amax, from frexp), the e4m3 cast of
    n * 2^-e, the entry assembled as bytes and scattered into the cache with
    index_copy_."""
    q, kv = ds["q"], ds["kv"]
    T = q.shape[0]
    cs = ds["cos_sin"].index_select(0, ds["positions"])
    c, s = cs[:, :32], cs[:, 32:]

    def norm_rope(x, w, cc, ss):
        n = torch.nn.functional.rms_norm(x.float(), (512,), w.float(), ds["eps"])
        e, o = n[..., 448::2], n[..., 449::2]
        n[..., 448:] = torch.stack([e * cc - o * ss, o * cc + e * ss], -1).flatten(-2)
        return n

    q.copy_(norm_rope(q, ds["q_weight"], c[:, None, :], s[:, None, :]).to(torch.bfloat16))
    n = norm_rope(kv, ds["kv_weight"], c, s)
    blocks = n[:, :448].view(T, 7, 64)
    amax = blocks.abs().amax(-1)
    mant, ex = torch.frexp(amax)                       # amax = mant * 2^ex, mant in [0.5, 1)
    e = ex - 9 + (mant > 0.875).to(ex.dtype)           # 448 = 0.875 * 2^9
    byte = torch.where(amax > 0, (e + 127).clamp(0, 254), torch.zeros_like(e))
    codes = torch.ldexp(blocks, (127 - byte)[..., None].to(torch.float32))
    codes = codes.to(torch.float8_e4m3fn).view(torch.uint8).view(T, 448)
    rope = n[:, 448:].to(torch.bfloat16).contiguous().view(torch.uint8)
    entry = torch.cat([codes, rope, byte.to(torch.uint8),
                       torch.zeros((T, 1), dtype=torch.uint8, device=q.device)], -1)
    slots = ds["slot_mapping"]
    keep = (slots >= 0).nonzero().squeeze(1)
    ds["kv_cache"].view(-1, ENTRY).index_copy_(0, slots.index_select(0, keep),
                                                entry.index_select(0, keep))


ENTRY = wl.ENTRY_BYTES


def time_unfused(qk, ds, reps, device):
    """Median ms of each unfused operator on the step's own inputs."""
    stream = torch.cuda.current_stream(device)
    out = {}
    for name, fn, d in (("qk", unfused_qk, qk), ("dsv4", unfused_dsv4, ds)):
        fn(d)
        torch.cuda.synchronize(device)
        med, _ = _time_launch(lambda: fn(d), reps, stream)
        out[name] = med
    return out


# ---------------------------------------------------------------------------
# every workload of the benchmark configurations, one record each
# ---------------------------------------------------------------------------

PER_CONFIG_L2_FLUSH_BELOW = 256 * 2**20


def config_workloads():
    """(config index, operator, workload) for every workload the benchmark
    configurations name: the packed-QKV decode and prefill cases, the DSV4
    decode and 32768-token cases, and each point of the DSV4 token sweep."""
    out = [(0, "qk", wl.QK_SMALL), (1, "qk", wl.QK_LARGE), (2, "dsv4", wl.DSV4_DECODE),
           (3, "dsv4", wl.DSV4_LARGE)]
    out += [(4, "dsv4", w) for w in wl.DSV4_SWEEP]
    return out


def oracle_gbs(op, d, sample_tokens):
    """The CPU oracle's GB/s on the first `sample_tokens` tokens of workload
    `d` (all host cores), by the same byte count as the GPU figure."""
    import oracle
    per_token = ("qkv", "positions") if op == "qk" else ("q", "kv", "positions", "slot_mapping")
    T = d[per_token[0]].shape[0]
    S = min(sample_tokens, T)

    def h(k):
        t = d[k][:S] if k in per_token else d[k]
        return wl.bf16_bits(t) if t.dtype == torch.bfloat16 else wl.host(t)
    if op == "qk":
        args = (h("qkv"), d["Hq"], d["Hk"], d["Hv"], d["D"], d["eps"], h("q_weight"),
                h("k_weight"), h("cos_sin"), h("positions"))
        t0 = time.perf_counter()
        oracle.qk_norm_rope(*args)
        dt = time.perf_counter() - t0
        nb = qk_bytes(S, d["Hq"], d["Hk"], d["D"])
    else:
        cache = h("kv_cache").copy()
        slots = h("slot_mapping")
        args = (h("q"), h("kv"), d["eps"], h("q_weight"), h("kv_weight"), h("cos_sin"),
                h("positions"), slots, cache)
        t0 = time.perf_counter()
        oracle.dsv4(*args)
        dt = time.perf_counter() - t0
        nb = dsv4_bytes(S, d["H"], int((slots >= 0).sum()))
    return nb / dt / 1e9, S


def per_config(kvq, device, peak, with_oracle=True, oracle_tokens=2048):
    """One record per configured workload under the automatic launch shape."""
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(512 * 2**20 // 4, dtype=torch.float32, device=device)
    recs = []
    for idx, op, w in config_workloads():
        if op == "qk":
            d = wl.make_qk_workload(w, device=device)
            nb = qk_bytes(w.T, w.Hq, w.Hk, w.D)
            fn = lambda: launch_qk(kvq, d, stream)  # noqa: E731
            shape = kvq.configs("qk")[kvq.qk_config_for(w.T, w.Hq, w.Hk)]
        else:
            d = wl.make_dsv4_workload(w, device=device)
            nb = dsv4_bytes(w.T, w.H, int((d["slot_mapping"] >= 0).sum()))
            fn = lambda: launch_dsv4(kvq, d, stream)  # noqa: E731
            shape = kvq.configs("dsv4")[kvq.dsv4_config_for(w.T, w.H)]
        small = nb < PER_CONFIG_L2_FLUSH_BELOW
        fn()
        torch.cuda.synchronize(device)
        reps = 30 if nb < 2**31 else 10
        med, best = _time_launch(fn, reps, stream, flush if small else None)
        rec = {"config": idx, "workload": w.name, "launch_shape": shape, "bytes": nb,
               "us_median": round(med * 1e3, 2), "gbs": round(nb / med / 1e6, 1),
               "pct_of_peak": round(100 * nb / med / 1e6 / peak, 2),
               "l2": "flushed between launches" if small else "larger than L2",
               "launches": reps}
        # the copy ceiling at this launch length: a plain device copy moving
        # the same bytes (half read, half written), timed the same way
        src = torch.empty(nb // 2, dtype=torch.uint8, device=device)
        dst = torch.empty_like(src)
        dst.copy_(src)
        cmed, _ = _time_launch(lambda: dst.copy_(src), reps, stream, flush if small else None)
        rec["copy_us_median"] = round(cmed * 1e3, 2)
        rec["pct_of_copy"] = round(100 * cmed / med, 1)
        del src, dst
        if with_oracle:
            g, S = oracle_gbs(op, d, oracle_tokens)
            rec["cpu_oracle_gbs"] = round(g, 3)
            rec["cpu_oracle_tokens"] = S
        recs.append(rec)
        del d
    del flush
    return recs


# ---------------------------------------------------------------------------
# the rows beyond the two operators' benchmarked layouts: cache read-back,
# other QK layouts, decode steps in a CUDA graph
# ---------------------------------------------------------------------------

def next_rows(kvq, device, peak):
    """One record per measured extension: dsv4_kv_cache_gather on random
    slots of a full 65536-slot cache; fused_qk_norm_rope at head_dim 64 and
    256 and with partial or GPT-J rotation; a 32-layer decode step (QK 17
    tokens + DSV4 16 tokens x 64 heads per layer) replayed as one CUDA graph."""
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(512 * 2**20 // 4, dtype=torch.float32, device=device)
    recs = []

    def copy_ceiling(rec, nb):
        # a plain device copy moving the same bytes, after the same flush
        src = torch.empty(nb // 2, dtype=torch.uint8, device=device)
        dst = torch.empty_like(src)
        dst.copy_(src)
        cmed, _ = _time_launch(lambda: dst.copy_(src), 30, stream, flush)
        rec["copy_us_median"] = round(cmed * 1e3, 2)
        rec["pct_of_copy"] = round(100 * cmed / (rec["us_median"] * 1e-3), 1)
        return rec

    d = wl.make_dsv4_workload(wl.DSV4_LARGE, device=device)
    launch_dsv4(kvq, d, stream)
    for n in (16, 32768, 131072):
        slots = torch.randint(0, 65536, (n,), device=device, dtype=torch.int64,
                              generator=torch.Generator(device=device).manual_seed(n))
        rows = torch.empty((n, 512), dtype=torch.bfloat16, device=device)
        nb = n * (584 + 8 + 1024)
        fn = lambda: kvq.dsv4_kv_cache_gather(d["kv_cache"], slots, rows, stream)  # noqa: E731
        fn()
        med, _ = _time_launch(fn, 30, stream, flush)
        recs.append(copy_ceiling({"row": "f2 dsv4_kv_cache_gather", "rows": n, "bytes": nb,
                                  "us_median": round(med * 1e3, 2),
                                  "gbs": round(nb / med / 1e6, 1),
                                  "pct_of_peak": round(100 * nb / med / 1e6 / peak, 2),
                                  "l2": "flushed between launches"}, nb))
    del d
    for T, D, rot, neox in ((32768, 64, 64, True), (32768, 64, 32, False), (32768, 128, 64, True),
                            (32768, 128, 128, False), (16384, 256, 256, True),
                            (16384, 256, 64, False)):
        q = wl.make_qk(T, 32, 8, 8, D=D, theta=1e6, max_pos=131072, seed=D + rot, device=device,
                       rotary_dim=rot, is_neox=neox)
        nb = qk_bytes(T, 32, 8, D, rot)
        fn = lambda: kvq.fused_qk_norm_rope(q["qkv"], 32, 8, 8, D, q["eps"], q["q_weight"],  # noqa: E731
                                            q["k_weight"], q["cos_sin"], neox, q["positions"],
                                            stream=stream, rotary_dim=rot)
        fn()
        med, _ = _time_launch(fn, 30, stream, flush)
        recs.append(copy_ceiling({
            "row": "f1 fused_qk_norm_rope_ex", "tokens": T, "heads": [32, 8, 8], "head_dim": D,
            "rotary_dim": rot, "pairs": "neox" if neox else "gptj", "bytes": nb,
            "us_median": round(med * 1e3, 2), "gbs": round(nb / med / 1e6, 1),
            "pct_of_peak": round(100 * nb / med / 1e6 / peak, 2),
            "l2": "flushed between launches (each launch follows a 512 MB write)"}, nb))
        del q
    layers = []
    for i in range(32):
        q = wl.make_qk(17, 16, 8, 8, theta=1e4, max_pos=4096, seed=i, device=device)
        ds = wl.make_dsv4(16, 64, max_pos=65536, num_blocks=64, block_size=64,
                          slots="distinct_skip2", seed=i, device=device)
        layers.append((q, ds))

    def decode(st):
        for q, ds in layers:
            launch_qk(kvq, q, st)
            launch_dsv4(kvq, ds, st)
    decode(stream)
    torch.cuda.synchronize(device)
    eager_ms, _ = _time_launch(lambda: decode(stream), 20, stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        decode(torch.cuda.current_stream(device))
    graph.replay()
    torch.cuda.synchronize(device)
    graph_ms, _ = _time_launch(graph.replay, 20, stream)
    recs.append({"row": "f3 decode step in a CUDA graph", "layers": 32,
                 "launches": 64, "eager_us": round(eager_ms * 1e3, 1),
                 "graph_us": round(graph_ms * 1e3, 1),
                 "graph_us_per_launch": round(graph_ms * 1e3 / 64, 2)})
    del graph, layers, flush
    return recs


def config_block(extra=None):
    c = {"workload": "fused_qk_norm_rope T=32768 Hq/Hk/Hv=32/8/8 D=128 theta=1e6 + "
                     "dsv4_qnorm_rope_kv_rope_quant_insert T=32768 H=64 (65536-slot cache)",
         "tokens_per_step": 32768, "qk_heads": [32, 8, 8], "dsv4_heads": 64,
         "l2": "inputs larger than L2 (qkv 403 MB, q 2.1 GB); no flush"}
    if extra:
        c.update(extra)
    return c


def run_gpu(args):
    import kv_quant_cache_gb300 as kvq
    world, rank, local = dist_setup()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    kvq.lib()
    qk, ds = make_step_inputs(device)
    b_qk, b_ds = step_bytes(qk, ds)
    host_inputs = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host_inputs = host_step_inputs(qk, ds)
    warmup = max(args.warmup, 3)
    clocks = ClockSampler(local)
    total_ms, qk_ms, ds_ms = time_device(kvq, qk, ds, args.steps, warmup, world, device)
    clk = clocks.stop()
    total_ms = max_over_ranks(total_ms, world, device)
    ms_step = total_ms / args.steps
    value = world * (b_qk + b_ds) / (ms_step * 1e-3) / 1e9
    peak, peak_kind = peak_hbm()
    ds_avg = statistics.mean(ds_ms)
    qk_avg = statistics.mean(qk_ms)
    achieved = b_ds / (ds_avg * 1e-3) / 1e9
    traffic = recorded_traffic("dsv4_stream_T32768_H64")
    e2e = None
    if not args.no_e2e:
        e2e_steps = max(1, args.steps if args.e2e_steps is None else args.e2e_steps)
        zc_ms, h2d, d2h = time_e2e_zero_copy(kvq, qk, ds, e2e_steps, device)
        zc_ms = max_over_ranks(zc_ms, world, device)
        st_ms, s_h2d, s_d2h, n_chunks = time_e2e(kvq, qk, ds, e2e_steps, device)
        st_ms = max_over_ranks(st_ms, world, device)
        e2e = {"value": round(world * (b_qk + b_ds) / (zc_ms * 1e-3) / 1e9, 2), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(zc_ms, 4), "steps": e2e_steps,
               "path": "C ABI called with pinned host buffers; the kernels read and write "
                       "them in place over NVLink-C2C (host->device / device->host bytes = "
                       "bytes the kernels read from / write to host memory); the paged cache "
                       "(in HBM) is copied back to pinned host memory every step",
               "staged_copies": {"value": round(world * (b_qk + b_ds) / (st_ms * 1e-3) / 1e9, 2),
                                 "ms_per_step": round(st_ms, 4), "h2d_bytes_per_step": s_h2d,
                                 "d2h_bytes_per_step": s_d2h,
                                 "pipeline": f"{n_chunks} token chunks, cudaMemcpyAsync in / "
                                             "kernels / out on three streams, steps handed "
                                             "over chunk by chunk"}}
    context = None
    per_cfg = None
    nexts = None
    if rank == 0 and not args.no_per_config:
        unf = time_unfused(qk, ds, 10, device)
        context = {"unfused_torch": {
            "what": "the step's two operators as separate eager PyTorch passes on this GPU "
                    "(rms_norm x2 + RoPE x2 for QK; rms_norm + RoPE of q and kv, blockwise "
                    "frexp/ldexp/e4m3 cast, entry assembly and index_copy_ for DSV4), fp32 "
                    "intermediates; GB/s by the same algorithmic bytes as the fused kernels",
            "qk_ms": round(unf["qk"], 4), "dsv4_ms": round(unf["dsv4"], 4),
            "qk_gbs": round(b_qk / (unf["qk"] * 1e-3) / 1e9, 1),
            "dsv4_gbs": round(b_ds / (unf["dsv4"] * 1e-3) / 1e9, 1),
            "step_gbs": round((b_qk + b_ds) / ((unf["qk"] + unf["dsv4"]) * 1e-3) / 1e9, 1),
            "fused_speedup": round((unf["qk"] + unf["dsv4"]) / ms_step, 2)}}
        per_cfg = per_config(kvq, device, peak, with_oracle=host_inputs is not None)
        nexts = next_rows(kvq, device, peak)
    cpu = None
    if host_inputs is not None:
        v, cores, dt = cpu_baseline(qk, ds, *host_inputs)
        v1, s1, dt1 = cpu_baseline_one_thread(qk, ds, *host_inputs)
        cpu = {"value": round(v, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "one whole step (both operators, all 32768 tokens, the same input "
                         "bytes as the GPU step), fp64 oracle, all host cores",
               "seconds": round(dt, 2),
               "one_thread": {"value": round(v1, 4), "unit": UNIT, "tokens": s1,
                              "seconds": round(dt1, 2),
                              "sample": f"the first {s1} tokens of each operator, one thread"}}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_block({
            "algorithmic_bytes_per_step": b_qk + b_ds, "qk_bytes": b_qk, "dsv4_bytes": b_ds,
            "qk_ms": round(qk_avg, 5), "dsv4_ms": round(ds_avg, 5),
            "kernel_times": "a second pass of the same steps with an event around each "
                            "launch (those events cost the launch overlap, so the step time "
                            "comes from the first pass, which has none)",
            "qk_gbs": round(b_qk / (qk_avg * 1e-3) / 1e9, 1),
            "core_bytes_per_step": core_bytes(qk, ds),
            "core_gbs": round(world * core_bytes(qk, ds) / (ms_step * 1e-3) / 1e9, 2),
            "core_bytes": "Q/K rows, q rows and kv vectors read, rows and cache entries "
                          "written; without cos/sin rows, positions, slots and weights",
            "qk_kernel": kvq.configs("qk")[kvq.qk_config_for(32768, 32, 8)],
            "pct_of_peak": round(100 * value / world / peak, 2),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}),
        "roofline": {"bound": "hbm",
                     "kernel": "dsv4 " + kvq.configs("dsv4")[kvq.dsv4_config_for(32768, 64)],
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "algorithmic_bytes_per_launch": b_ds},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 2 * args.steps, "clocks": clk,
        "gpu_launches_note": "launches in the timed region; the per-kernel pass launches as "
                             "many again",
        "per_config": per_cfg, "next_rows": nexts, "context": context,
        "dispatch": {"qk": kvq.configs("qk")[kvq.qk_config_for(32768, 32, 8)],
                     "dsv4": kvq.configs("dsv4")[kvq.dsv4_config_for(32768, 64)]},
    }
    if args.sweep and rank == 0:
        sweep(kvq, device)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------

def _reference_inputs(S):
    """Host inputs of the benchmarked step's two workloads at S tokens (the
    same recipes and seeds, drawn by the CPU generator)."""
    qk = wl.make_qk(S, 32, 8, 8, theta=1e6, max_pos=131072, seed=1001)
    ds = wl.make_dsv4(S, 64, max_pos=131072, num_blocks=1024, block_size=64,
                      slots="perm_prefix", seed=1003)
    host = {k: (wl.bf16_bits(v) if v.dtype == torch.bfloat16 else wl.host(v))
            for k, v in {**{"qkv": qk["qkv"], "qw": qk["q_weight"], "kw": qk["k_weight"],
                            "cs1": qk["cos_sin"], "p1": qk["positions"]},
                         **{"q": ds["q"], "dqw": ds["q_weight"], "dkw": ds["kv_weight"],
                            "kv": ds["kv"], "cs2": ds["cos_sin"], "p2": ds["positions"],
                            "slot": ds["slot_mapping"], "cache": ds["kv_cache"]}}.items()}
    return host, qk["eps"], ds["eps"]


def _reference_step(h, eps_qk, eps_ds):
    import oracle
    oracle.qk_norm_rope(h["qkv"], 32, 8, 8, 128, eps_qk, h["qw"], h["kw"], h["cs1"], h["p1"],
                        out=h["qkv"])
    oracle.dsv4(h["q"], h["kv"], eps_ds, h["dqw"], h["dkw"], h["cs2"], h["p2"], h["slot"],
                h["cache"], q_out=h["q"])


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on the host cores,
    doing the benchmarked step (both operators, all 32768 tokens) per step.
    Only when K + W such steps would not finish within --reference-budget-s
    does each step take a token sample of the workload instead (stated in
    the line)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    T = wl.QK_LARGE.T
    warmup = max(args.warmup, 3)
    S = args.cpu_sample_tokens
    if S is None:
        probe, e1, e2 = _reference_inputs(1024)
        _reference_step(probe, e1, e2)
        t0 = time.perf_counter()
        _reference_step(probe, e1, e2)
        per_token = (time.perf_counter() - t0) / 1024
        fit = int(args.reference_budget_s / ((args.steps + warmup) * per_token))
        S = max(64, min(T, fit // 64 * 64))
        del probe
    S = max(1, min(S, T))
    h, eps_qk, eps_ds = _reference_inputs(S)
    for _ in range(warmup):
        _reference_step(h, eps_qk, eps_ds)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _reference_step(h, eps_qk, eps_ds)
    dt = (time.perf_counter() - t0) / args.steps
    nbytes = qk_bytes(S, 32, 8) + dsv4_bytes(S, 64, S)
    value = nbytes / dt / 1e9
    sample = ("the whole step: both operators, all 32768 tokens" if S == T else
              f"first {S} of 32768 tokens of both operators per step (the requested steps "
              f"at full size would exceed {args.reference_budget_s:.0f} s)")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": config_block({"tokens_per_step_processed": S, "same_config": S == T,
                                "l2": "host memory (CPU oracle)"}),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "kind": "oracle",
                         "cores": oracle.default_threads(), "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# sweep: every parity workload, both launch shapes, copy ceiling
# ---------------------------------------------------------------------------

def _time_launch(fn, reps, stream, flush=None):
    times = []
    for _ in range(reps):
        if flush is not None:
            flush.add_(1)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    ms = sorted(x.elapsed_time(y) for x, y in times)
    return ms[len(ms) // 2], ms[0]


def sweep(kvq, device):
    """Every workload under every launch configuration, the DSV4 dispatch
    crossover, a 512 MiB device-to-device copy ceiling and the pinned-host
    link's copy ceiling (JSON lines on stderr)."""
    peak, _ = peak_hbm()
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(512 * 2**20 // 4, dtype=torch.float32, device=device)
    out = []

    def emit(rec):
        out.append(rec)
        sys.stderr.write(json.dumps(rec) + "\n")
        sys.stderr.flush()

    src = torch.empty(512 * 2**20, dtype=torch.uint8, device=device)
    dst = torch.empty_like(src)
    med, best = _time_launch(lambda: dst.copy_(src), 20, stream)
    emit({"sweep": "d2d_copy_512MiB", "gbs_median": round(2 * src.numel() / med / 1e6, 1),
          "gbs_best": round(2 * src.numel() / best / 1e6, 1)})
    del src, dst
    # host-link ceiling for the end-to-end figures: 1 GiB pinned host <-> HBM
    # copies, each direction alone, then both at once on two streams
    h_in = torch.empty(2**30, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(2**30, dtype=torch.uint8, pin_memory=True)
    d_in = torch.empty(2**30, dtype=torch.uint8, device=device)
    d_out = torch.empty(2**30, dtype=torch.uint8, device=device)
    side = torch.cuda.Stream(device)

    def both():
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            h_out.copy_(d_out, non_blocking=True)
        d_in.copy_(h_in, non_blocking=True)
        stream.wait_stream(side)
    with torch.cuda.stream(stream):
        t_h2d, _ = _time_launch(lambda: d_in.copy_(h_in, non_blocking=True), 5, stream)
        t_d2h, _ = _time_launch(lambda: h_out.copy_(d_out, non_blocking=True), 5, stream)
        t_both, _ = _time_launch(both, 5, stream)
    emit({"sweep": "host_link_1GiB", "h2d_gbs": round(2**30 / t_h2d / 1e6, 1),
          "d2h_gbs": round(2**30 / t_d2h / 1e6, 1),
          "both_gbs": round(2 * 2**30 / t_both / 1e6, 1)})
    del h_in, h_out, d_in, d_out

    def run_configs(op, name, nb, fn, reps):
        small = nb < 256 * 2**20
        auto = None
        for cid, cname in [(-1, "auto")] + list(enumerate(kvq.configs(op))):
            old = kvq.set_config(op, cid)
            try:
                med, _ = _time_launch(fn, reps, stream, flush if small else None)
            finally:
                kvq.set_config(op, old)
            emit({"sweep": name, "config": cname, "bytes": nb, "us_median": round(med * 1e3, 2),
                  "gbs": round(nb / med / 1e6, 1), "pct_peak": round(100 * nb / med / 1e6 / peak, 1),
                  "l2_flush": small})

    for w in (wl.QK_SMALL, wl.QK_LARGE,
              wl.QKWorkload("qk_T131072_32-8-8", T=131072, Hq=32, Hk=8, Hv=8, theta=1e6,
                            max_pos=131072, seed=1001)):
        d = wl.make_qk_workload(w, device=device)
        run_configs("qk", w.name, qk_bytes(w.T, w.Hq, w.Hk), lambda: launch_qk(kvq, d, stream), 30)
        del d
    # QK launch-shape crossover: the small-batch, register-pipelined and
    # TMA-staged shapes of the head_dim-128 kernel over the token count
    names = kvq.configs("qk")
    cand = [names.index(n) for n in ("tiles<4w,1step>", "tiles<4w,4step>") if n in names]
    cand += [i for i, n in enumerate(names) if n.startswith("bulk")]
    for T in (1, 16, 64, 256, 1024, 2048, 4096, 8192, 16384, 65536):
        d = wl.make_qk(T, 32, 8, 8, theta=1e6, max_pos=131072, seed=5 + T, device=device)
        nb = qk_bytes(T, 32, 8)
        small = nb < 256 * 2**20
        res = {}
        for cid in cand:
            old = kvq.set_config("qk", cid)
            try:
                res[names[cid]] = round(_time_launch(lambda: launch_qk(kvq, d, stream), 30, stream,
                                                     flush if small else None)[0] * 1e3, 2)
            finally:
                kvq.set_config("qk", old)
        emit({"sweep": "qk_dispatch", "T": T, "rows": T * 40, "bytes": nb, "us": res,
              "auto": names[kvq.qk_config_for(T, 32, 8)]})
        del d
    # the copy ceiling by launch length: a device copy moving (read + write)
    # the given traffic, for comparison with any kernel of the same bytes
    for mb in (64, 128, 256, 512, 1024, 2048, 4096, 8192):
        src = torch.empty(mb * 2**19, dtype=torch.uint8, device=device)
        dst = torch.empty_like(src)
        med, _ = _time_launch(lambda: dst.copy_(src), 20, stream,
                              flush if mb < 256 else None)
        emit({"sweep": "d2d_copy_ceiling", "traffic_mb": mb, "us_median": round(med * 1e3, 2),
              "gbs": round(mb * 2**20 / med / 1e6, 1),
              "pct_peak": round(100 * mb * 2**20 / med / 1e6 / peak, 1)})
        del src, dst
    # the same crossover for two general layouts: one-shot general kernel vs
    # the staged shape
    gen = names.index("general<frag4>")
    stg = names.index("bulk<16w,2st,6KB>")
    for D, rot, neox in ((64, 64, True), (256, 64, False)):
        for T in (1024, 4096, 8192, 16384, 32768):
            d = wl.make_qk(T, 32, 8, 8, D=D, theta=1e6, max_pos=131072, seed=9 + T, device=device,
                           rotary_dim=rot, is_neox=neox)
            nb = qk_bytes(T, 32, 8, D, rot)
            res = {}
            for cid in (gen, stg):
                old = kvq.set_config("qk", cid)
                try:
                    res[names[cid]] = round(_time_launch(
                        lambda: kvq.fused_qk_norm_rope(d["qkv"], 32, 8, 8, D, d["eps"],
                                                       d["q_weight"], d["k_weight"], d["cos_sin"],
                                                       neox, d["positions"], stream=stream,
                                                       rotary_dim=rot),
                        30, stream, flush if nb < 256 * 2**20 else None)[0] * 1e3, 2)
                finally:
                    kvq.set_config("qk", old)
            emit({"sweep": "qk_dispatch_general", "D": D, "rot": rot, "neox": neox, "T": T,
                  "rows": T * 40, "bytes": nb, "us": res})
            del d
    # a copy moving the QK step's bytes (Q+K rows read and written): the
    # ceiling for a launch of that length
    nb = qk_bytes(wl.QK_LARGE.T, wl.QK_LARGE.Hq, wl.QK_LARGE.Hk)
    src = torch.empty(nb // 2, dtype=torch.uint8, device=device)
    dst = torch.empty_like(src)
    med, _ = _time_launch(lambda: dst.copy_(src), 30, stream)
    emit({"sweep": "d2d_copy_qk_T32768_bytes", "bytes": nb, "us_median": round(med * 1e3, 2),
          "gbs": round(nb / med / 1e6, 1), "pct_peak": round(100 * nb / med / 1e6 / peak, 1)})
    del src, dst
    # the general QK layouts (head_dim 64/256, GPT-J pairs, partial rotation):
    # the automatic choice, both one-shot fragment widths and the staged shapes
    general = [(i, n) for i, n in enumerate(kvq.configs("qk"))
               if n.startswith("general") or n.startswith("bulk")]
    for (T, hq, hk, hv, D, rot, neox) in ((32768, 32, 8, 8, 64, 64, True),
                                          (32768, 32, 8, 8, 64, 32, False),
                                          (32768, 32, 8, 8, 128, 64, True),
                                          (32768, 32, 8, 8, 128, 64, False),
                                          (32768, 32, 8, 8, 128, 128, False),
                                          (16384, 32, 8, 8, 256, 256, True),
                                          (16384, 32, 8, 8, 256, 64, False),
                                          (17, 16, 8, 8, 256, 256, True)):
        d = wl.make_qk(T, hq, hk, hv, D=D, theta=1e6, max_pos=131072, seed=D + rot,
                       device=device, rotary_dim=rot, is_neox=neox)
        nb = qk_bytes(T, hq, hk, D, rot)
        small = nb < 256 * 2**20

        def fn():
            kvq.fused_qk_norm_rope(d["qkv"], hq, hk, hv, D, d["eps"], d["q_weight"],
                                   d["k_weight"], d["cos_sin"], neox, d["positions"],
                                   stream=stream, rotary_dim=rot)
        for cid, cname in [(-1, "auto")] + general:
            old = kvq.set_config("qk", cid)
            try:
                med, _ = _time_launch(fn, 30, stream, flush if small else None)
            finally:
                kvq.set_config("qk", old)
            emit({"sweep": f"qk_T{T}_{hq}-{hk}-{hv}_D{D}_rot{rot}_{'neox' if neox else 'gptj'}",
                  "config": cname, "bytes": nb, "us_median": round(med * 1e3, 2),
                  "gbs": round(nb / med / 1e6, 1),
                  "pct_peak": round(100 * nb / med / 1e6 / peak, 1), "l2_flush": small})
        del d
    for w in [wl.DSV4_DECODE, wl.DSV4_LARGE, *wl.DSV4_SWEEP]:
        d = wl.make_dsv4_workload(w, device=device)
        nb = dsv4_bytes(w.T, w.H, int((d["slot_mapping"] >= 0).sum()))
        run_configs("dsv4", w.name, nb, lambda: launch_dsv4(kvq, d, stream), 30 if nb < 2**32 else 8)
        del d
    # reading entries back: random slots of a full 65536-slot cache
    for n in (16, 32768, 131072):
        d = wl.make_dsv4_workload(wl.DSV4_LARGE, device=device)
        launch_dsv4(kvq, d, stream)
        slots = torch.randint(0, 65536, (n,), device=device, dtype=torch.int64)
        rows = torch.empty((n, 512), dtype=torch.bfloat16, device=device)
        nb = n * (584 + 8 + 1024)
        small = nb < 256 * 2**20
        med, _ = _time_launch(lambda: kvq.dsv4_kv_cache_gather(d["kv_cache"], slots, rows, stream),
                              30, stream, flush if small else None)
        emit({"sweep": f"gather_n{n}", "config": "gather", "bytes": nb,
              "us_median": round(med * 1e3, 2), "gbs": round(nb / med / 1e6, 1),
              "pct_peak": round(100 * nb / med / 1e6 / peak, 1), "l2_flush": small})
        del d
    # decode step: 32 layers of (QK 17 tokens + DSV4 16 tokens x 64 heads),
    # eager launches vs one CUDA graph replay
    layers = []
    for i in range(32):
        qk = wl.make_qk(17, 16, 8, 8, theta=1e4, max_pos=4096, seed=i, device=device)
        ds = wl.make_dsv4(16, 64, max_pos=65536, num_blocks=64, block_size=64,
                          slots="distinct_skip2", seed=i, device=device)
        layers.append((qk, ds))

    def decode_step(st):
        for qk, ds in layers:
            launch_qk(kvq, qk, st)
            launch_dsv4(kvq, ds, st)
    for pdl in (False, True):
        old = kvq.set_programmatic_launch(pdl)
        try:
            decode_step(stream)
            torch.cuda.synchronize()
            eager_ms, _ = _time_launch(lambda: decode_step(stream), 20, stream)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                decode_step(torch.cuda.current_stream(device))
            graph.replay()
            torch.cuda.synchronize()
            graph_ms, _ = _time_launch(graph.replay, 20, stream)
        finally:
            kvq.set_programmatic_launch(old)
        emit({"sweep": "decode_32_layers", "programmatic_launch": pdl,
              "eager_us": round(eager_ms * 1e3, 1), "graph_us": round(graph_ms * 1e3, 1),
              "eager_us_per_launch": round(eager_ms * 1e3 / 64, 2),
              "graph_us_per_launch": round(graph_ms * 1e3 / 64, 2)})
        del graph
    del layers
    # the benchmarked step, and a mid-size step (QK 4096 tokens + DSV4 2048
    # tokens x 64 heads), with and without programmatic dependent launch
    mid = (wl.make_qk(4096, 32, 8, 8, theta=1e6, max_pos=131072, seed=3, device=device),
           wl.make_dsv4(2048, 64, max_pos=131072, num_blocks=64, block_size=64, seed=4,
                        device=device))
    for name, (qk, ds) in (("step", make_step_inputs(device)), ("step_mid", mid)):
        nb = sum(step_bytes(qk, ds))
        for pdl in (False, True):
            old = kvq.set_programmatic_launch(pdl)
            try:
                def step():
                    launch_qk(kvq, qk, stream)
                    launch_dsv4(kvq, ds, stream)
                step()
                med, _ = _time_launch(step, 50, stream, flush if nb < 256 * 2**20 else None)
            finally:
                kvq.set_programmatic_launch(old)
            emit({"sweep": name, "programmatic_launch": pdl, "bytes": nb,
                  "us_median": round(med * 1e3, 2), "gbs": round(nb / med / 1e6, 1),
                  "pct_peak": round(100 * nb / med / 1e6 / peak, 1)})
        del qk, ds
    del mid
    # dispatch crossover between the small- and large-batch shapes
    for H in (64, 128):
        for T in (1, 4, 16, 64, 128, 256, 512, 1024, 4096):
            d = wl.make_dsv4(T, H, max_pos=131072, num_blocks=-(-2 * T // 64), block_size=64,
                             seed=7 + T, device=device)
            res = {}
            for path, thr in (("small", 1 << 40), ("large", 0)):
                old = kvq.set_dsv4_dispatch_threshold(thr)
                try:
                    res[path] = _time_launch(lambda: launch_dsv4(kvq, d, stream), 30, stream, flush)[0]
                finally:
                    kvq.set_dsv4_dispatch_threshold(old)
            emit({"sweep": "dispatch", "T": T, "H": H, "programs": T * (H + 1),
                  "small_us": round(res["small"] * 1e3, 2), "large_us": round(res["large"] * 1e3, 2)})
            del d
    return out


def run_profile_case(args):
    """A reduced case of one kernel for profiler captures: --profile qk|dsv4,
    --tokens T, --heads H, --launches n (each launch on the same inputs),
    --shape NAME (a launch shape by its name; default: the automatic one);
    for qk also --head-dim, --rotary-dim (default: the head dim) and --gptj."""
    import kv_quant_cache_gb300 as kvq
    device = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(device)
    if args.shape is not None:
        names = kvq.configs(args.profile)
        if args.shape not in names:
            raise SystemExit(f"--shape: {args.shape!r} is not one of {names}")
        kvq.set_config(args.profile, names.index(args.shape))
    if args.profile == "qk":
        D = args.head_dim
        rot = D if args.rotary_dim is None else args.rotary_dim
        d = wl.make_qk(args.tokens, args.heads, 8, 8, D=D, theta=1e6, max_pos=131072, seed=1001,
                       device=device, rotary_dim=rot, is_neox=not args.gptj)
        fn = lambda: kvq.fused_qk_norm_rope(  # noqa: E731
            d["qkv"], args.heads, 8, 8, D, d["eps"], d["q_weight"], d["k_weight"], d["cos_sin"],
            not args.gptj, d["positions"], stream=stream, rotary_dim=rot)
        nb = qk_bytes(args.tokens, args.heads, 8, D, rot)
    else:
        d = wl.make_dsv4(args.tokens, args.heads, max_pos=131072,
                         num_blocks=-(-2 * args.tokens // 64), block_size=64, seed=1003,
                         device=device)
        fn, nb = (lambda: launch_dsv4(kvq, d, stream)), dsv4_bytes(args.tokens, args.heads, args.tokens)
    fn()  # the first call does the per-device set-up; time the later ones
    torch.cuda.synchronize(device)
    med, best = _time_launch(fn, args.launches, stream)
    print(json.dumps({"profile": args.profile, "tokens": args.tokens, "heads": args.heads,
                      "bytes": nb, "us_median": round(med * 1e3, 2),
                      "gbs": round(nb / med / 1e6, 1)}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("kvq", "reference"), default="kvq")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="steps of the end-to-end legs (default: --steps)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload records and the unfused PyTorch context")
    ap.add_argument("--cpu-sample-tokens", type=int, default=None,
                    help="tokens per step of the reference (oracle) arm (default: all 32768, "
                         "fewer only if the requested steps would not finish within "
                         "--reference-budget-s)")
    ap.add_argument("--reference-budget-s", type=float, default=90.0)
    ap.add_argument("--profile", choices=("qk", "dsv4"), default=None)
    ap.add_argument("--tokens", type=int, default=4096)
    ap.add_argument("--heads", type=int, default=64)
    ap.add_argument("--launches", type=int, default=5)
    ap.add_argument("--shape", default=None)
    ap.add_argument("--head-dim", type=int, default=128)
    ap.add_argument("--rotary-dim", type=int, default=None)
    ap.add_argument("--gptj", action="store_true")
    args = ap.parse_args()
    if args.profile:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
