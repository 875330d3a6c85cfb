"""GB300 (sm_103a) attention-prologue kernels -- Python binding of include/kvq.h.

This module only marshals arguments: it checks that tensors are CUDA tensors
(or pinned host tensors, which the kernels then access in place over the
host interconnect) of the expected dtype and layout, takes their addresses
and the current stream, and calls the C ABI in ``libkvq.so``.  Every step of the computation
runs in the CUDA kernels; there is no CPU or PyTorch fallback.  If the library
has not been built, importing works but every call raises ``KvqError``.

Build: ``python -m kv_quant_cache_gb300._build`` (or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

import torch

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libkvq.so")

KVQ_OK = 0
KVQ_ERR_NULL = 1
KVQ_ERR_SHAPE = 2
KVQ_ERR_UNSUPPORTED = 3
KVQ_ERR_ALIGN = 4
KVQ_ERR_CUDA = 5
KVQ_ERR_VALUE = 6

ENTRY_BYTES = 584
DSV4_DIM = 512
DSV4_ROPE_DIM = 64  # rotated dims of a DSV4 row: cos/sin table width


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(what)
        self.status = status


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_F = ctypes.c_float


def _declare(L: ctypes.CDLL) -> ctypes.CDLL:
    L.fused_qk_norm_rope.restype = _I
    L.fused_qk_norm_rope.argtypes = [_P, _I64, _I, _I, _I, _I, _F, _P, _P, _P, _I, _P, _P]
    L.fused_qk_norm_rope_ex.restype = _I
    L.fused_qk_norm_rope_ex.argtypes = [_P, _I64, _I, _I, _I, _I, _F, _P, _P, _P, _I, _I, _P,
                                        _P]
    L.dsv4_qnorm_rope_kv_rope_quant_insert.restype = _I
    L.dsv4_qnorm_rope_kv_rope_quant_insert.argtypes = [_P, _P, _I64, _I, _F, _P, _P, _P, _P,
                                                       _P, _P, _I, _P]
    L.dsv4_qnorm_rope_kv_rope_quant_insert_out.restype = _I
    L.dsv4_qnorm_rope_kv_rope_quant_insert_out.argtypes = [_P, _P, _P, _I64, _I, _F, _P, _P,
                                                           _P, _P, _P, _P, _I, _P]
    L.fused_qk_norm_rope_checked.restype = _I
    L.fused_qk_norm_rope_checked.argtypes = [_P, _I64, _I, _I, _I, _I, _F, _P, _P, _P, _I64, _I,
                                             _I, _P, _P, _P]
    L.dsv4_qnorm_rope_kv_rope_quant_insert_checked.restype = _I
    L.dsv4_qnorm_rope_kv_rope_quant_insert_checked.argtypes = [_P, _P, _P, _I64, _I, _F, _P, _P,
                                                               _P, _I64, _P, _P, _P, _I64, _I,
                                                               _P, _P]
    L.dsv4_kv_cache_gather_checked.restype = _I
    L.dsv4_kv_cache_gather_checked.argtypes = [_P, _I64, _I, _P, _I64, _P, _P, _P]
    L.dsv4_kv_cache_gather.restype = _I
    L.dsv4_kv_cache_gather.argtypes = [_P, _I, _P, _I64, _P, _P]
    L.kvq_status_string.restype = ctypes.c_char_p
    L.kvq_status_string.argtypes = [_I]
    L.kvq_last_cuda_error.restype = _I
    L.kvq_last_cuda_error.argtypes = []
    L.kvq_dsv4_dispatch_threshold.restype = _I64
    L.kvq_dsv4_dispatch_threshold.argtypes = []
    L.kvq_set_dsv4_dispatch_threshold.restype = _I64
    L.kvq_set_dsv4_dispatch_threshold.argtypes = [_I64]
    L.kvq_dsv4_dispatch_path.restype = _I
    L.kvq_dsv4_dispatch_path.argtypes = [_I64, _I]
    for op in ("qk", "dsv4"):
        getattr(L, f"kvq_{op}_num_configs").restype = _I
        getattr(L, f"kvq_{op}_num_configs").argtypes = []
        getattr(L, f"kvq_{op}_config_name").restype = ctypes.c_char_p
        getattr(L, f"kvq_{op}_config_name").argtypes = [_I]
        getattr(L, f"kvq_set_{op}_config").restype = _I
        getattr(L, f"kvq_set_{op}_config").argtypes = [_I]
    L.kvq_qk_config_for.restype = _I
    L.kvq_qk_config_for.argtypes = [_I64, _I, _I]
    L.kvq_set_stage_wait_limit.restype = ctypes.c_uint32
    L.kvq_set_stage_wait_limit.argtypes = [ctypes.c_uint32]
    L.kvq_stage_events.restype = _I
    L.kvq_stage_events.argtypes = [_P, _P, _I]
    L.kvq_set_programmatic_launch.restype = _I
    L.kvq_set_programmatic_launch.argtypes = [_I]
    L.kvq_dsv4_config_for.restype = _I
    L.kvq_dsv4_config_for.argtypes = [_I64, _I]
    return L


_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises KvqError if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise KvqError(-1, f"{LIB_PATH} not found: build it with "
                               "`python -m kv_quant_cache_gb300._build`")
        _LIB = _declare(ctypes.CDLL(LIB_PATH))
    return _LIB


def status_string(status: int) -> str:
    return lib().kvq_status_string(status).decode()


def _check(status: int, fn: str) -> None:
    if status != KVQ_OK:
        msg = f"{fn}: {status_string(status)}"
        if status == KVQ_ERR_CUDA:
            msg += f" (cudaError {lib().kvq_last_cuda_error()})"
        raise KvqError(status, msg)


def _cuda(t: torch.Tensor, dtype, name: str) -> int:
    """Address of a CUDA tensor, or of a pinned host tensor (mapped into the
    device's address space at the same address under unified addressing)."""
    if type(t) is torch.Tensor and t.is_cuda and t.dtype == dtype and t.is_contiguous():
        return t.data_ptr()  # the common case, checked first (per-call cost)
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or (t.device.type == "cpu"
                                                             and t.is_pinned())):
        raise ValueError(f"{name}: expected a CUDA tensor or a pinned host tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    return t.data_ptr()


# torch's current raw stream handle without building a Stream object (a few
# times cheaper per call); the public API is the fallback.
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device) -> int:
    """Raw handle of ``stream`` (default: torch's current stream of ``device``,
    a CUDA device index; -1 = the current device)."""
    if stream is None:
        if _raw_current_stream is not None and device >= 0:
            return _raw_current_stream(device)
        stream = torch.cuda.current_stream(device if device >= 0 else None)
    if hasattr(stream, "cuda_stream"):
        sd = getattr(stream, "device", None)
        if device >= 0 and sd is not None and sd.index is not None and sd.index != device:
            raise ValueError(f"stream is on cuda:{sd.index}, the tensors on cuda:{device}")
        return stream.cuda_stream
    return int(stream)


# The current device as torch's runtime sees it (the raw query, without the
# public API's lazy-initialisation check; the public API is the fallback).
_current_device = getattr(torch._C, "_cuda_getDevice", None) or torch.cuda.current_device


def _device(*tensors) -> int:
    """The one CUDA device that every CUDA tensor of a call is on (pinned host
    tensors, whose get_device() is -1, may take part on any device); -1 if
    none is a CUDA tensor."""
    dev = -1
    for t in tensors:
        if t is not None:
            d = t.get_device()
            if d != dev and d >= 0:
                if dev >= 0:
                    raise ValueError(f"tensors on cuda:{dev} and cuda:{d}: every CUDA tensor "
                                     "of one call must be on the same device")
                dev = d
    return dev


def _on(dev, fn, *args):
    """Call the C entry point ``fn`` with ``dev`` as the current device: the
    library launches on, and keeps its per-device set-up for, the current
    device, so a call whose tensors live on another GPU switches to it."""
    if dev >= 0 and dev != _current_device():
        with torch.cuda.device(dev):
            return fn(*args)
    return fn(*args)


def _counter(errors, name="errors"):
    return _cuda(errors, torch.int32, name)


def fused_qk_norm_rope(qkv, num_heads_q, num_heads_k, num_heads_v, head_dim, eps,
                       q_weight, k_weight, cos_sin_cache, is_neox, positions,
                       stream=None, rotary_dim=None, errors=None) -> None:
    """In-place per-head RMSNorm + RoPE of the Q and K heads of ``qkv``.

    qkv: bf16 [T, (Hq+Hk+Hv)*head_dim]; weights bf16 [head_dim]; cos_sin_cache
    fp32 [max_pos, rotary_dim]; positions int64 [T].  Same parameter order as
    the C entry point (stream last, default: torch's current stream).
    ``rotary_dim`` (default: the cos/sin table's width) selects partial
    rotation through ``fused_qk_norm_rope_ex``; ``is_neox`` picks NeoX (True)
    or GPT-J (False) pairs.  ``errors`` (an int32 CUDA tensor, zeroed by the
    caller) selects the bounds-checked launch: tokens whose position is
    outside the table are left unchanged and counted there.
    """
    if qkv.dim() != 2 or qkv.shape[1] != (num_heads_q + num_heads_k + num_heads_v) * head_dim:
        raise ValueError("qkv must be [T, (Hq+Hk+Hv)*head_dim]")
    if rotary_dim is None:
        rotary_dim = cos_sin_cache.shape[1]
    if cos_sin_cache.dim() != 2 or cos_sin_cache.shape[1] != rotary_dim:
        raise ValueError("cos_sin_cache must be [max_pos, rotary_dim]")
    T = qkv.shape[0]
    if q_weight.numel() != head_dim or k_weight.numel() != head_dim:
        raise ValueError("q_weight and k_weight must hold head_dim values")
    if positions.numel() != T:
        raise ValueError("positions must hold one value per token")
    dev = _device(qkv, q_weight, k_weight, cos_sin_cache, positions, errors)
    args = (_cuda(qkv, torch.bfloat16, "qkv"), T, num_heads_q, num_heads_k, num_heads_v,
            head_dim, float(eps), _cuda(q_weight, torch.bfloat16, "q_weight"),
            _cuda(k_weight, torch.bfloat16, "k_weight"),
            _cuda(cos_sin_cache, torch.float32, "cos_sin_cache"))
    tail = (int(rotary_dim), int(bool(is_neox)), _cuda(positions, torch.int64, "positions"))
    if errors is None:
        st = _on(dev, lib().fused_qk_norm_rope_ex, *args, *tail, _stream(stream, dev))
    else:
        st = _on(dev, lib().fused_qk_norm_rope_checked, *args, cos_sin_cache.shape[0], *tail,
                 _counter(errors), _stream(stream, dev))
    _check(st, "fused_qk_norm_rope")


def dsv4_qnorm_rope_kv_rope_quant_insert(q, kv, eps, q_weight, kv_weight, cos_sin_cache,
                                         positions, slot_mapping, kv_cache,
                                         stream=None, q_out=None, errors=None) -> None:
    """DSV4 prologue: q [T,H,512] normalised + rotated (in place, or into
    ``q_out`` when given); the kv vectors [T,512] normalised, rotated,
    quantised and written to ``kv_cache`` uint8 [num_blocks, block_size, 584]
    at ``slot_mapping``.  ``errors`` (int32 CUDA tensor, zeroed by the caller)
    selects the bounds-checked launch: tokens with a position outside the
    table or a slot outside the cache are rejected and counted there."""
    if q.dim() != 3 or q.shape[2] != DSV4_DIM:
        raise ValueError("q must be [T, H, 512]")
    if kv.dim() != 2 or kv.shape[0] != q.shape[0] or kv.shape[1] != DSV4_DIM:
        raise ValueError("kv must be [T, 512]")
    if kv_cache.dim() != 3 or kv_cache.shape[2] != ENTRY_BYTES:
        raise ValueError("kv_cache must be [num_blocks, block_size, 584]")
    T, H = q.shape[0], q.shape[1]
    if q_out is None:
        q_out = q
    if q_out.shape != q.shape:
        raise ValueError("q_out must have q's shape")
    if q_weight.numel() != DSV4_DIM or kv_weight.numel() != DSV4_DIM:
        raise ValueError("q_weight and kv_weight must hold 512 values")
    if cos_sin_cache.dim() != 2 or cos_sin_cache.shape[1] != DSV4_ROPE_DIM:
        raise ValueError("cos_sin_cache must be [max_pos, 64]")
    if positions.numel() != T or slot_mapping.numel() != T:
        raise ValueError("positions and slot_mapping must hold one value per token")
    dev = _device(q, q_out, kv, q_weight, kv_weight, cos_sin_cache, positions, slot_mapping,
                  kv_cache, errors)
    head = (_cuda(q, torch.bfloat16, "q"), _cuda(q_out, torch.bfloat16, "q_out"),
            _cuda(kv, torch.bfloat16, "kv"), T, H, float(eps),
            _cuda(q_weight, torch.bfloat16, "q_weight"),
            _cuda(kv_weight, torch.bfloat16, "kv_weight"),
            _cuda(cos_sin_cache, torch.float32, "cos_sin_cache"))
    idx = (_cuda(positions, torch.int64, "positions"),
           _cuda(slot_mapping, torch.int64, "slot_mapping"), _cuda(kv_cache, torch.uint8, "kv_cache"))
    if errors is None:
        st = _on(dev, lib().dsv4_qnorm_rope_kv_rope_quant_insert_out, *head, *idx,
                 kv_cache.shape[1], _stream(stream, dev))
    else:
        st = _on(dev, lib().dsv4_qnorm_rope_kv_rope_quant_insert_checked,
                 *head, cos_sin_cache.shape[0], *idx, kv_cache.shape[0], kv_cache.shape[1],
                 _counter(errors), _stream(stream, dev))
    _check(st, "dsv4_qnorm_rope_kv_rope_quant_insert")


def dsv4_kv_cache_gather(kv_cache, slots, out=None, stream=None, errors=None):
    """bf16 [n, 512] rows read back from the cache entries at ``slots``
    (int64 [n], -1 = a zero row); ``out`` is allocated if not given.
    ``errors`` (int32 CUDA tensor) selects the bounds-checked launch."""
    if kv_cache.dim() != 3 or kv_cache.shape[2] != ENTRY_BYTES:
        raise ValueError("kv_cache must be [num_blocks, block_size, 584]")
    if slots.dim() != 1:
        raise ValueError("slots must be a 1-D int64 tensor")
    n = slots.shape[0]
    if out is None:
        out = torch.empty((n, DSV4_DIM), dtype=torch.bfloat16, device=kv_cache.device)
    if out.shape != (n, DSV4_DIM):
        raise ValueError("out must be [len(slots), 512]")
    dev = _device(kv_cache, slots, out, errors)
    if errors is None:
        st = _on(dev, lib().dsv4_kv_cache_gather,
                 _cuda(kv_cache, torch.uint8, "kv_cache"), kv_cache.shape[1],
                 _cuda(slots, torch.int64, "slots"), n, _cuda(out, torch.bfloat16, "out"),
                 _stream(stream, dev))
    else:
        st = _on(dev, lib().dsv4_kv_cache_gather_checked,
                 _cuda(kv_cache, torch.uint8, "kv_cache"), kv_cache.shape[0], kv_cache.shape[1],
                 _cuda(slots, torch.int64, "slots"), n, _cuda(out, torch.bfloat16, "out"),
                 _counter(errors), _stream(stream, dev))
    _check(st, "dsv4_kv_cache_gather")
    return out


def dsv4_dispatch_threshold() -> int:
    return lib().kvq_dsv4_dispatch_threshold()


def set_dsv4_dispatch_threshold(value: int) -> int:
    """Set the DSV4 program-count threshold (< 0 restores the default); returns the old one."""
    return lib().kvq_set_dsv4_dispatch_threshold(int(value))


def dsv4_dispatch_path(num_tokens: int, num_heads: int) -> int:
    return lib().kvq_dsv4_dispatch_path(int(num_tokens), int(num_heads))


def configs(op: str) -> list:
    """Names of the launch configurations of ``op`` ("qk" or "dsv4")."""
    L = lib()
    n = getattr(L, f"kvq_{op}_num_configs")()
    return [getattr(L, f"kvq_{op}_config_name")(i).decode() for i in range(n)]


def set_config(op: str, config_id: int) -> int:
    """Force launch configuration ``config_id`` of ``op`` (< 0: automatic);
    returns the previous override."""
    prev = getattr(lib(), f"kvq_set_{op}_config")(int(config_id))
    if prev == -2:
        raise ValueError(f"{op}: no launch configuration {config_id}")
    return prev


def set_stage_wait_limit(polls: int) -> int:
    """Polls of a stage barrier before a warp of a staged QK launch shape
    finishes from global memory (0: always); returns the previous limit."""
    return lib().kvq_set_stage_wait_limit(int(polls))


def stage_events(reset: bool = False) -> tuple:
    """(fallbacks, drain_timeouts) counted by the staged QK launch shapes on
    the current device since the last reset (waits for the device first)."""
    fb, dt = ctypes.c_uint64(0), ctypes.c_uint64(0)
    _check(lib().kvq_stage_events(ctypes.addressof(fb), ctypes.addressof(dt), int(bool(reset))),
           "kvq_stage_events")
    return fb.value, dt.value


def set_programmatic_launch(enable: bool) -> bool:
    """Launch later kernels with programmatic stream serialization (the
    default: they may be scheduled while the previous kernel finishes; results
    are unchanged); returns the previous setting."""
    return bool(lib().kvq_set_programmatic_launch(1 if enable else 0))


def qk_config_for(num_tokens: int, num_heads_q: int, num_heads_k: int) -> int:
    return lib().kvq_qk_config_for(int(num_tokens), int(num_heads_q), int(num_heads_k))


def dsv4_config_for(num_tokens: int, num_heads: int) -> int:
    return lib().kvq_dsv4_config_for(int(num_tokens), int(num_heads))
