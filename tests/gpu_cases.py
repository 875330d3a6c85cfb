"""Run the CUDA path and the oracle on the same seeded inputs and compare.

Used by the ``-m gpu`` tests.  Inputs come from ``workloads`` (seeded); the
CUDA side is called through the C ABI (``kv_quant_cache_gb300``); the
expected values come from ``oracle`` only.  Large workloads are compared in
token slices (the operators are per-token independent, so slicing is exact).
"""
from __future__ import annotations

import numpy as np
import torch

import kv_quant_cache_gb300 as kvq
import oracle
import workloads as wl
from parity import Bf16Report, CacheReport, compare_cache


def to_device(d, dev):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


# ---------------------------------------------------------------------------
# packed-QKV operator
# ---------------------------------------------------------------------------

def qk_parity(d, slice_tokens=4096, call=None) -> Bf16Report:
    """d: inputs on the GPU (make_qk ... device=cuda).  Runs the op in place,
    then compares every token with the oracle.  V must be bit-identical."""
    Hq, Hk, Hv, D = d["Hq"], d["Hk"], d["Hv"], d["D"]
    rot, neox = d.get("rot", D), d.get("is_neox", True)
    qkv_in = d["qkv"].clone()
    if call is None:
        kvq.fused_qk_norm_rope(d["qkv"], Hq, Hk, Hv, D, d["eps"], d["q_weight"], d["k_weight"],
                               d["cos_sin"], neox, d["positions"], rotary_dim=rot)
    else:
        call(d)
    torch.cuda.synchronize()
    qw, kw = wl.bf16_bits(d["q_weight"]), wl.bf16_bits(d["k_weight"])
    cs, pos = wl.host(d["cos_sin"]), wl.host(d["positions"])
    T = qkv_in.shape[0]
    NR = Hq + Hk
    rep = Bf16Report()
    for a in range(0, T, slice_tokens):
        b = min(T, a + slice_tokens)
        inp = wl.bf16_bits(qkv_in[a:b])
        gpu = wl.bf16_bits(d["qkv"][a:b]).reshape(b - a, NR + Hv, D)
        out, ref, mag = oracle.qk_norm_rope(inp, Hq, Hk, Hv, D, d["eps"], qw, kw, cs,
                                            np.ascontiguousarray(pos[a:b]), is_neox=neox,
                                            rot_dim=rot, want_ref=True)
        assert np.array_equal(gpu[:, NR:], inp.reshape(b - a, NR + Hv, D)[:, NR:]), "V changed"
        rep.add(gpu[:, :NR], out.reshape(b - a, NR + Hv, D)[:, :NR], ref, mag)
    rep.check("fused_qk_norm_rope")
    return rep


def qk_parity_sampled(d, sample, seed=0, call=None) -> Bf16Report:
    """Like qk_parity for workloads too large to compare whole: the first and
    last 8 tokens and `sample` random ones against the oracle; V checked
    bit-identical for every token on the GPU."""
    Hq, Hk, Hv, D = d["Hq"], d["Hk"], d["Hv"], d["D"]
    rot, neox = d.get("rot", D), d.get("is_neox", True)
    T = d["qkv"].shape[0]
    NR = Hq + Hk
    qkv_in = d["qkv"].clone()
    if call is None:
        kvq.fused_qk_norm_rope(d["qkv"], Hq, Hk, Hv, D, d["eps"], d["q_weight"], d["k_weight"],
                               d["cos_sin"], neox, d["positions"], rotary_dim=rot)
    else:
        call(d)
    torch.cuda.synchronize()
    v_cols = slice(NR * D, (NR + Hv) * D)
    assert torch.equal(d["qkv"][:, v_cols], qkv_in[:, v_cols]), "V changed"
    rng = np.random.default_rng(seed)
    idx = np.unique(np.concatenate([np.arange(min(8, T)), np.arange(max(T - 8, 0), T),
                                    rng.choice(T, size=min(sample, T), replace=False)]))
    idx_t = torch.from_numpy(idx).to(d["qkv"].device)
    inp = wl.bf16_bits(qkv_in.index_select(0, idx_t))
    gpu = wl.bf16_bits(d["qkv"].index_select(0, idx_t)).reshape(idx.size, NR + Hv, D)
    out, ref, mag = oracle.qk_norm_rope(inp, Hq, Hk, Hv, D, d["eps"], wl.bf16_bits(d["q_weight"]),
                                        wl.bf16_bits(d["k_weight"]), wl.host(d["cos_sin"]),
                                        np.ascontiguousarray(wl.host(d["positions"])[idx]),
                                        is_neox=neox, rot_dim=rot, want_ref=True)
    rep = Bf16Report()
    rep.add(gpu[:, :NR], out.reshape(idx.size, NR + Hv, D)[:, :NR], ref, mag)
    rep.check("fused_qk_norm_rope")
    return rep


# ---------------------------------------------------------------------------
# DSV4 operator
# ---------------------------------------------------------------------------

def run_dsv4(d):
    kvq.dsv4_qnorm_rope_kv_rope_quant_insert(d["q"], d["kv"], d["eps"], d["q_weight"],
                                             d["kv_weight"], d["cos_sin"], d["positions"],
                                             d["slot_mapping"], d["kv_cache"])


def dsv4_parity(d, slice_tokens=2048, sample=None, seed=0, call=None):
    """Run the op on d (GPU tensors) and compare with the oracle.

    sample=None: every token, whole cache compared (bytes outside mapped
    entries bit-exact).  sample=n: n tokens (first, last and random ones); the
    sampled tokens' q rows and cache entries are compared, and the rest of the
    cache is checked for the sentinel on the GPU.
    ``call(d)`` replaces the library call (the unfused baseline's test).
    Returns (q report, cache report)."""
    T = d["q"].shape[0]
    q_in = d["q"].clone()
    cache_in = d["kv_cache"].clone()
    (call or run_dsv4)(d)
    torch.cuda.synchronize()
    qw, kvw = wl.bf16_bits(d["q_weight"]), wl.bf16_bits(d["kv_weight"])
    cs = wl.host(d["cos_sin"])
    if sample is None or sample >= T:
        idx = np.arange(T)
    else:
        rng = np.random.default_rng(seed)
        idx = np.unique(np.concatenate([np.arange(min(8, T)), np.arange(max(T - 8, 0), T),
                                        rng.choice(T, size=sample, replace=False)]))
    idx_t = torch.from_numpy(idx).to(d["q"].device)
    pos = wl.host(d["positions"])[idx]
    slots = wl.host(d["slot_mapping"])[idx]
    kv = wl.bf16_bits(d["kv"].index_select(0, idx_t))
    ora_cache = wl.host(cache_in).copy()
    qrep = Bf16Report()
    kv_ref = np.empty((idx.size, 512))
    kv_mag = np.empty((idx.size, 512))
    margin = np.empty((idx.size, 7))
    for a in range(0, idx.size, slice_tokens):
        b = min(idx.size, a + slice_tokens)
        sel = idx_t[a:b]
        res = oracle.dsv4(wl.bf16_bits(q_in.index_select(0, sel)), np.ascontiguousarray(kv[a:b]),
                          d["eps"], qw, kvw, cs, np.ascontiguousarray(pos[a:b]),
                          np.ascontiguousarray(slots[a:b]), ora_cache, want_ref=True)
        qrep.add(wl.bf16_bits(d["q"].index_select(0, sel)), res["q"], res["q_ref"], res["q_mag"])
        kv_ref[a:b], kv_mag[a:b], margin[a:b] = res["kv_ref"], res["kv_mag"], res["exp_margin"]
    qrep.check("dsv4 q")
    full = idx.size == T
    gpu_cache = wl.host(d["kv_cache"])
    crep = compare_cache(gpu_cache, ora_cache, slots, kv_ref, kv_mag, margin,
                         check_untouched=full)
    crep.check("dsv4 cache")
    if not full:
        untouched_sentinel_on_gpu(d["kv_cache"], cache_in, d["slot_mapping"])
    return qrep, crep


def untouched_sentinel_on_gpu(cache, cache_in, slot_mapping):
    """Every slot that no token maps to keeps its original bytes."""
    c = cache.view(-1, wl.ENTRY_BYTES)
    c0 = cache_in.view(-1, wl.ENTRY_BYTES)
    unmapped = torch.ones(c.shape[0], dtype=torch.bool, device=c.device)
    s = slot_mapping[slot_mapping >= 0]
    unmapped[s] = False
    assert torch.equal(c[unmapped], c0[unmapped]), "bytes outside mapped entries changed"
    written = c[~unmapped]
    assert int((written[:, 583] != 0).sum()) == 0, "pad byte of a written entry is not 0"


def with_threshold(value):
    """Context manager forcing the DSV4 dispatch threshold."""
    class _Ctx:
        def __enter__(self):
            self.old = kvq.set_dsv4_dispatch_threshold(value)

        def __exit__(self, *exc):
            kvq.set_dsv4_dispatch_threshold(self.old)
    return _Ctx()


def with_config(op, config_id):
    """Context manager forcing launch configuration ``config_id`` of ``op``."""
    class _Ctx:
        def __enter__(self):
            self.old = kvq.set_config(op, config_id)

        def __exit__(self, *exc):
            kvq.set_config(op, self.old)
    return _Ctx()


SMALL_PATH = 1 << 40   # threshold above any program count: small-batch launch
TILED_PATH = 0         # every call takes the token-tiled launch
