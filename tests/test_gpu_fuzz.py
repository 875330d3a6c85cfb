"""Seeded random cases across shapes, layouts, launch shapes and pointer
kinds, every one compared with the oracle.  The seed fixes the case list, so a
failure is reproducible by its id."""
import numpy as np
import pytest
import torch

import kv_quant_cache_gb300 as kvq
import workloads as wl
from gpu_cases import dsv4_parity, qk_parity, with_config, with_threshold

pytestmark = pytest.mark.gpu


def _qk_cases(n=100, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        D = int(rng.choice([64, 128, 256]))
        rot = int(rng.choice([r for r in range(16, D + 1, 16)]))
        neox = bool(rng.integers(2))
        T = int(rng.choice([1, 2, 3, 5, 8, 13, 31, 64, 100, 257, 1000, 3001]))
        Hq, Hk, Hv = (int(x) for x in rng.integers(0, 9, size=3))
        if Hq + Hk == 0:
            Hq = 1
        # every shape for the head_dim-128 full-NeoX layout; otherwise the
        # automatic choice, the one-shot general kernel or a staged shape
        names = kvq.configs("qk")
        choices = [-1] + [c for c, n in enumerate(names)
                          if (D, rot, neox) == (128, 128, True) or n.startswith(("general", "bulk"))]
        forced = int(rng.choice(choices))
        out.append((i, T, Hq, Hk, Hv, D, rot, neox, forced))
    return out


@pytest.mark.parametrize("case", _qk_cases(), ids=lambda c: f"qk{c[0]}")
def test_qk_random(cuda_device, case):
    i, T, Hq, Hk, Hv, D, rot, neox, forced = case
    d = wl.make_qk(T, Hq, Hk, Hv, D=D, theta=float(10 ** (3 + i % 4)), max_pos=8192,
                   seed=10_000 + i, device=cuda_device, rotary_dim=rot, is_neox=neox)
    with with_config("qk", forced):
        qk_parity(d)


def _dsv4_cases(n=80, seed=2025):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        T = int(rng.choice([1, 2, 3, 7, 16, 33, 100, 511, 1500, 4097]))
        H = int(rng.choice([1, 2, 3, 8, 16, 64, 128]))
        bs = int(rng.choice([1, 16, 64, 128]))
        nb = -(-int(rng.integers(T, 3 * T + 2)) // bs)
        forced = int(rng.integers(-1, len(kvq.configs("dsv4"))))
        host = bool(rng.integers(4) == 0)
        out.append((i, T, H, bs, nb, forced, host))
    return out


@pytest.mark.parametrize("case", _dsv4_cases(), ids=lambda c: f"dsv4_{c[0]}")
def test_dsv4_random(cuda_device, case):
    i, T, H, bs, nb, forced, host = case
    d = wl.make_dsv4(T, H, max_pos=131072, num_blocks=nb, block_size=bs,
                     slots="distinct_skip2", seed=20_000 + i, device=cuda_device)
    if host:  # activations in pinned host memory, read in place by the kernels
        for k in ("q", "kv", "positions", "slot_mapping"):
            d[k] = d[k].cpu().pin_memory()
    with with_config("dsv4", forced):
        dsv4_parity(d)


def test_gather_random(cuda_device):
    import oracle
    rng = np.random.default_rng(7)
    d = wl.make_dsv4(600, 4, max_pos=4096, num_blocks=20, block_size=64, seed=31,
                     device=cuda_device)
    kvq.dsv4_qnorm_rope_kv_rope_quant_insert(d["q"], d["kv"], d["eps"], d["q_weight"],
                                             d["kv_weight"], d["cos_sin"], d["positions"],
                                             d["slot_mapping"], d["kv_cache"])
    for n in (1, 7, 333, 5000):
        slots = torch.from_numpy(rng.integers(-1, 20 * 64, size=n)).to(cuda_device)
        out = kvq.dsv4_kv_cache_gather(d["kv_cache"], slots)
        torch.cuda.synchronize()
        want = oracle.dsv4_gather(wl.host(d["kv_cache"]), wl.host(slots))
        assert np.array_equal(wl.bf16_bits(out), want)
