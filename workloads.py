"""Seeded synthetic inputs for the attention-prologue operators.

Input recipes only: shapes, value distributions, index patterns and the rotary
cos/sin table that the model side would hand to the operators.  Nothing in this
module performs any step of the operators themselves (no normalisation, no
rotation, no quantisation, no cache packing), so the CUDA path and the CPU
oracle share nothing but the bytes produced here.

Recipe (every config, unless stated otherwise):
  * activations (qkv, q, kv): N(0, 1) rounded to bf16;
  * norm weights: N(1, 0.1) rounded to bf16;
  * eps = 1e-6;
  * cos/sin table: row p = [cos(p f_0..f_{R/2-1}), sin(p f_0..)], f_i =
    theta^(-2i/R), computed in fp64 and rounded once to fp32;
  * the paged cache is pre-filled with the sentinel byte 0xA5 so that any
    stray write shows up;
  * seed = 1000 + index of the workload in the list below.

Large tensors are drawn on the device they are needed on (torch's generator
for that device), small ones on the CPU; either way both sides of a parity
check receive the same bytes.
"""
from __future__ import annotations

import functools
import math
from dataclasses import dataclass, field

import numpy as np
import torch

ENTRY_BYTES = 584
DSV4_DIM = 512
SENTINEL = 0xA5
EPS = 1e-6


# ---------------------------------------------------------------------------
# Workload descriptions
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class QKWorkload:
    name: str
    T: int
    Hq: int
    Hk: int
    Hv: int
    D: int = 128
    theta: float = 1e4
    max_pos: int = 4096
    positions: str = "uniform"  # "arange" | "uniform"
    seed: int = 0


@dataclass(frozen=True)
class DSV4Workload:
    name: str
    T: int
    H: int
    theta: float = 1e4
    max_pos: int = 131072
    num_blocks: int = 1024
    block_size: int = 64
    slots: str = "distinct"  # "distinct" | "distinct_skip2" | "perm_prefix"
    seed: int = 0


# packed-QKV operator: a decode-sized case and a prefill-sized case
QK_SMALL = QKWorkload("qk_T17_16-8-8", T=17, Hq=16, Hk=8, Hv=8, theta=1e4,
                      max_pos=4096, positions="arange", seed=1000)
QK_LARGE = QKWorkload("qk_T32768_32-8-8", T=32768, Hq=32, Hk=8, Hv=8, theta=1e6,
                      max_pos=131072, positions="uniform", seed=1001)

# DSV4 operator: decode size, a large prefill, and a token sweep
DSV4_DECODE = DSV4Workload("dsv4_T16_H64", T=16, H=64, theta=1e4, max_pos=65536,
                           num_blocks=1024, block_size=64, slots="distinct_skip2",
                           seed=1002)
DSV4_LARGE = DSV4Workload("dsv4_T32768_H64", T=32768, H=64, theta=1e4, max_pos=131072,
                          num_blocks=1024, block_size=64, slots="perm_prefix", seed=1003)


def _sweep():
    out = []
    for i, T in enumerate((1, 17, 1024, 2048, 8192, 32768, 131072)):
        out.append(DSV4Workload(f"dsv4_T{T}_H128", T=T, H=128, max_pos=131072,
                                num_blocks=-(-2 * T // 64), block_size=64,
                                slots="distinct", seed=1004 + i))
    out.append(DSV4Workload("dsv4_T131072_H64", T=131072, H=64, max_pos=131072,
                            num_blocks=-(-2 * 131072 // 64), block_size=64,
                            slots="distinct", seed=1011))
    return tuple(out)


DSV4_SWEEP = _sweep()


# ---------------------------------------------------------------------------
# Generators
# ---------------------------------------------------------------------------

@functools.lru_cache(maxsize=8)
def _cos_sin_np(max_pos: int, rot_dim: int, theta: float) -> np.ndarray:
    half = rot_dim // 2
    inv = float(theta) ** (-(2.0 * np.arange(half, dtype=np.float64)) / rot_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.ascontiguousarray(
        np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32))


def cos_sin_table(max_pos: int, rot_dim: int, theta: float, device="cpu") -> torch.Tensor:
    """fp32 [max_pos, rot_dim]: cosines of the rot_dim/2 frequencies, then sines."""
    return torch.from_numpy(_cos_sin_np(max_pos, rot_dim, theta)).to(device)


def _gen(seed: int, device) -> torch.Generator:
    return torch.Generator(device=device).manual_seed(seed)


def _normal_bf16(shape, g, device, mean=0.0, std=1.0) -> torch.Tensor:
    x = torch.empty(shape, dtype=torch.bfloat16, device=device)
    x.normal_(mean, std, generator=g)
    return x


def make_qk(T, Hq, Hk, Hv, D=128, theta=1e4, max_pos=4096, positions="uniform",
            seed=0, device="cpu", eps=EPS, rotary_dim=None, is_neox=True):
    """Inputs of the packed-QKV operator as a dict of tensors on ``device``.
    The cos/sin table has ``rotary_dim`` columns (default: the head dim)."""
    rot = D if rotary_dim is None else rotary_dim
    g = _gen(seed, device)
    qkv = _normal_bf16((T, (Hq + Hk + Hv) * D), g, device)
    q_weight = _normal_bf16((D,), g, device, 1.0, 0.1)
    k_weight = _normal_bf16((D,), g, device, 1.0, 0.1)
    if positions == "arange":
        pos = torch.arange(T, dtype=torch.int64, device=device)
    else:
        pos = torch.randint(0, max_pos, (T,), generator=g, device=device, dtype=torch.int64)
    return dict(qkv=qkv, q_weight=q_weight, k_weight=k_weight,
                cos_sin=cos_sin_table(max_pos, rot, theta, device), positions=pos,
                Hq=Hq, Hk=Hk, Hv=Hv, D=D, eps=eps, rot=rot, is_neox=is_neox)


def make_qk_workload(w: QKWorkload, device="cpu"):
    return make_qk(w.T, w.Hq, w.Hk, w.Hv, w.D, w.theta, w.max_pos, w.positions,
                   w.seed, device)


def _slots(kind, T, n_slots, g, device):
    if kind == "perm_prefix" or kind == "distinct":
        if T > n_slots:
            raise ValueError("more tokens than cache slots")
        return torch.randperm(n_slots, generator=g, device=device)[:T].to(torch.int64)
    if kind == "distinct_skip2":
        s = torch.randperm(n_slots, generator=g, device=device)[:T].to(torch.int64)
        if T >= 2:
            idx = torch.randperm(T, generator=g, device=device)[:2]
            s[idx] = -1
        return s
    raise ValueError(kind)


def make_dsv4(T, H, theta=1e4, max_pos=131072, num_blocks=1024, block_size=64,
              slots="distinct", seed=0, device="cpu", eps=EPS):
    """Inputs of the DSV4 operator as a dict of tensors on ``device``."""
    g = _gen(seed, device)
    q = _normal_bf16((T, H, DSV4_DIM), g, device)
    kv = _normal_bf16((T, DSV4_DIM), g, device)
    q_weight = _normal_bf16((DSV4_DIM,), g, device, 1.0, 0.1)
    kv_weight = _normal_bf16((DSV4_DIM,), g, device, 1.0, 0.1)
    pos = torch.randint(0, max_pos, (T,), generator=g, device=device, dtype=torch.int64)
    slot_mapping = _slots(slots, T, num_blocks * block_size, g, device)
    kv_cache = torch.full((num_blocks, block_size, ENTRY_BYTES), SENTINEL,
                          dtype=torch.uint8, device=device)
    return dict(q=q, kv=kv, q_weight=q_weight, kv_weight=kv_weight,
                cos_sin=cos_sin_table(max_pos, 64, theta, device), positions=pos,
                slot_mapping=slot_mapping, kv_cache=kv_cache, H=H,
                block_size=block_size, eps=eps)


def make_dsv4_workload(w: DSV4Workload, device="cpu"):
    return make_dsv4(w.T, w.H, w.theta, w.max_pos, w.num_blocks, w.block_size,
                     w.slots, w.seed, device)


# ---------------------------------------------------------------------------
# torch <-> numpy views used to hand the same bytes to the oracle
# ---------------------------------------------------------------------------

def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 numpy view of a bf16 tensor (copied to the host if needed)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()


def bf16_from_values(values, device="cpu") -> torch.Tensor:
    return torch.as_tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16).to(device)
