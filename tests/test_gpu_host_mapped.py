"""Both operators on pinned host buffers (the kernels access them in place
through the device's mapping of host memory), against the oracle."""
import pytest
import torch

import kv_quant_cache_gb300 as kvq
import workloads as wl
from gpu_cases import dsv4_parity, qk_parity

pytestmark = pytest.mark.gpu


def _pinned(d, keys):
    return {k: (v.pin_memory() if k in keys else v) for k, v in d.items()}


@pytest.mark.parametrize("config", [-1, 7], ids=["auto", "bulk"])
def test_qk_on_pinned_host_buffers(cuda_device, config):
    """Also with a TMA-staged shape forced: the bulk-copy engine is only given
    device memory, so pinned buffers take the register-pipelined shape."""
    d = wl.make_qk(2048, 32, 8, 8, theta=1e6, max_pos=131072, seed=41, device="cpu")
    d = {k: (v.to(cuda_device) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    d["qkv"] = d["qkv"].cpu().pin_memory()
    d["positions"] = d["positions"].cpu().pin_memory()
    old = kvq.set_config("qk", config)
    try:
        qk_parity(d)
    finally:
        kvq.set_config("qk", old)


def test_dsv4_on_pinned_host_buffers(cuda_device):
    d = wl.make_dsv4(1024, 64, max_pos=131072, num_blocks=32, block_size=64, seed=42,
                     device=cuda_device)
    for k in ("q", "kv", "positions", "slot_mapping"):
        d[k] = d[k].cpu().pin_memory()
    qrep, crep = dsv4_parity(d)
    assert crep.entries == 1024


def test_pageable_host_tensor_is_rejected(cuda_device):
    d = wl.make_qk(4, 2, 1, 1, device="cpu")
    g = {k: (v.to(cuda_device) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    with pytest.raises(ValueError):
        kvq.fused_qk_norm_rope(d["qkv"], 2, 1, 1, 128, 1e-6, g["q_weight"], g["k_weight"],
                               g["cos_sin"], True, g["positions"])
