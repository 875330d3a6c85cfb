"""Bounds-checked entry points on the GPU.

Out-of-range positions and slots are passed on purpose here: the checked
kernels test every index against the sizes they are given before using it,
so such tokens are rejected and counted, never read or written out of range.
"""
import numpy as np
import pytest
import torch

import kv_quant_cache_gb300 as kvq
import oracle
import workloads as wl
from gpu_cases import run_dsv4, with_threshold, SMALL_PATH, TILED_PATH
from parity import Bf16Report, compare_cache

pytestmark = pytest.mark.gpu


def _clone(d):
    return {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _counter(dev):
    return torch.zeros(1, dtype=torch.int32, device=dev)


def _qk_call(d, errors=None):
    kvq.fused_qk_norm_rope(d["qkv"], d["Hq"], d["Hk"], d["Hv"], d["D"], d["eps"], d["q_weight"],
                           d["k_weight"], d["cos_sin"], d["is_neox"], d["positions"],
                           rotary_dim=d["rot"], errors=errors)


@pytest.mark.parametrize("layout", [(128, 128, True, 17), (128, 128, True, 3000),
                                    (256, 64, False, 500), (64, 64, True, 40)])
def test_qk_checked_equals_unchecked_on_valid_input(cuda_device, layout):
    D, rot, neox, T = layout
    d = wl.make_qk(T, 8, 2, 2, D=D, max_pos=4096, seed=61, device=cuda_device,
                   rotary_dim=rot, is_neox=neox)
    a, b = _clone(d), _clone(d)
    err = _counter(cuda_device)
    _qk_call(a)
    _qk_call(b, err)
    torch.cuda.synchronize()
    assert torch.equal(a["qkv"], b["qkv"]) and int(err.item()) == 0


@pytest.mark.parametrize("layout", [(128, 128, True), (256, 128, False)])
def test_qk_checked_rejects_bad_positions(cuda_device, layout):
    D, rot, neox = layout
    T, Hq, Hk, Hv, P = 300, 6, 2, 2, 1024
    d = wl.make_qk(T, Hq, Hk, Hv, D=D, max_pos=P, seed=62, device=cuda_device,
                   rotary_dim=rot, is_neox=neox)
    pos = wl.host(d["positions"]).copy()
    bad = np.zeros(T, bool)
    bad[[0, 7, 150, 299]] = True
    pos[[0, 7, 150, 299]] = [P, -1, 10**12, P + 5]
    d["positions"] = torch.from_numpy(pos).to(cuda_device)
    qkv_in = wl.bf16_bits(d["qkv"])
    err = _counter(cuda_device)
    _qk_call(d, err)
    torch.cuda.synchronize()
    assert int(err.item()) == int(bad.sum())
    got = wl.bf16_bits(d["qkv"])
    assert np.array_equal(got[bad], qkv_in[bad])                      # left unchanged
    good = ~bad
    out, ref, mag = oracle.qk_norm_rope(np.ascontiguousarray(qkv_in[good]), Hq, Hk, Hv, D, d["eps"],
                                        wl.bf16_bits(d["q_weight"]), wl.bf16_bits(d["k_weight"]),
                                        wl.host(d["cos_sin"]), np.ascontiguousarray(pos[good]),
                                        is_neox=neox, rot_dim=rot, want_ref=True)
    NR = Hq + Hk
    g3 = got[good].reshape(-1, NR + Hv, D)
    rep = Bf16Report()
    rep.add(g3[:, :NR], out.reshape(-1, NR + Hv, D)[:, :NR], ref, mag)
    rep.check("checked qk")


@pytest.mark.parametrize("threshold", [SMALL_PATH, TILED_PATH], ids=["small", "large"])
def test_dsv4_checked_equals_unchecked_on_valid_input(cuda_device, threshold):
    d = wl.make_dsv4(2048, 8, max_pos=8192, num_blocks=64, block_size=64,
                     slots="distinct_skip2", seed=63, device=cuda_device)
    a, b = _clone(d), _clone(d)
    err = _counter(cuda_device)
    with with_threshold(threshold):
        run_dsv4(a)
        kvq.dsv4_qnorm_rope_kv_rope_quant_insert(b["q"], b["kv"], b["eps"], b["q_weight"],
                                                 b["kv_weight"], b["cos_sin"], b["positions"],
                                                 b["slot_mapping"], b["kv_cache"], errors=err)
    torch.cuda.synchronize()
    assert torch.equal(a["q"], b["q"]) and torch.equal(a["kv_cache"], b["kv_cache"])
    assert int(err.item()) == 0


@pytest.mark.parametrize("threshold", [SMALL_PATH, TILED_PATH], ids=["small", "large"])
def test_dsv4_checked_rejects_bad_positions_and_slots(cuda_device, threshold):
    T, H, P, nb, bs = 1000, 4, 2048, 40, 64
    d = wl.make_dsv4(T, H, max_pos=P, num_blocks=nb, block_size=bs, slots="distinct",
                     seed=64, device=cuda_device)
    pos = wl.host(d["positions"]).copy()
    slots = wl.host(d["slot_mapping"]).copy()
    bad_pos = np.zeros(T, bool)
    bad_slot = np.zeros(T, bool)
    bad_pos[[3, 500, 999]] = True
    pos[[3, 500, 999]] = [-7, P, 2**40]
    bad_slot[[10, 11, 700]] = True
    slots[[10, 11, 700]] = [nb * bs, -2, 2**50]
    slots[[20, 21]] = -1                                   # no slot: not an error
    d["positions"] = torch.from_numpy(pos).to(cuda_device)
    d["slot_mapping"] = torch.from_numpy(slots).to(cuda_device)
    q_in, cache_in = wl.bf16_bits(d["q"]), wl.host(d["kv_cache"]).copy()
    err = _counter(cuda_device)
    with with_threshold(threshold):
        kvq.dsv4_qnorm_rope_kv_rope_quant_insert(d["q"], d["kv"], d["eps"], d["q_weight"],
                                                 d["kv_weight"], d["cos_sin"], d["positions"],
                                                 d["slot_mapping"], d["kv_cache"], errors=err)
    torch.cuda.synchronize()
    assert int(err.item()) == int((bad_pos | bad_slot).sum())
    q_gpu = wl.bf16_bits(d["q"])
    assert np.array_equal(q_gpu[bad_pos], q_in[bad_pos])   # rows of bad positions untouched
    ok = ~bad_pos
    o_slots = np.where(bad_slot, -1, slots)[ok]           # rejected slots: no entry expected
    o_cache = cache_in.copy()
    res = oracle.dsv4(np.ascontiguousarray(q_in[ok]), np.ascontiguousarray(wl.bf16_bits(d["kv"])[ok]),
                      d["eps"], wl.bf16_bits(d["q_weight"]), wl.bf16_bits(d["kv_weight"]),
                      wl.host(d["cos_sin"]), np.ascontiguousarray(pos[ok]),
                      np.ascontiguousarray(o_slots), o_cache, want_ref=True)
    rep = Bf16Report()
    rep.add(q_gpu[ok], res["q"], res["q_ref"], res["q_mag"])
    rep.check("checked dsv4 q")
    compare_cache(wl.host(d["kv_cache"]), o_cache, o_slots, res["kv_ref"], res["kv_mag"],
                  res["exp_margin"]).check("checked dsv4 cache")


def test_gather_checked(cuda_device):
    d = wl.make_dsv4(100, 2, max_pos=1024, num_blocks=4, block_size=64, seed=65, device=cuda_device)
    run_dsv4(d)
    slots = torch.tensor([0, 255, 256, -1, -3, 17, 2**40], dtype=torch.int64, device=cuda_device)
    err = _counter(cuda_device)
    out = kvq.dsv4_kv_cache_gather(d["kv_cache"], slots, errors=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 3
    s = wl.host(slots)
    want = oracle.dsv4_gather(wl.host(d["kv_cache"]), np.where((s >= 0) & (s < 256), s, -1))
    assert np.array_equal(wl.bf16_bits(out), want)
