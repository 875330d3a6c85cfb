"""CPU fp64 oracle for the attention-prologue operators.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product package
(``kv_quant_cache_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, one token at a time; see
the header comment of ``oracle.h`` for the sources and readings).  This module
only compiles that file with gcc, loads it with ctypes and marshals numpy
arrays.  bf16 tensors are passed as their uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
SO_PATH = os.path.join(_HERE, "liboracle.so")

DSV4_DIM = 512
DSV4_ENTRY = 584
DSV4_NBLOCK = 7


class OracleError(RuntimeError):
    pass


def build(force: bool = False, src: str = _SRC, out: str = SO_PATH, defines=()) -> str:
    """Compile ``oracle.c`` into a shared library (skipped when up to date)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= max(os.path.getmtime(src), os.path.getmtime(_HDR))):
        return out
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
           "-I", _HERE, *[f"-D{d}" for d in defines], src, "-o", tmp, "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
    except subprocess.CalledProcessError as e:
        os.unlink(tmp)
        raise OracleError(f"oracle build failed:\n{e.stderr}") from e
    os.replace(tmp, out)
    return out


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    lib.orc_bf16_value.restype = ctypes.c_double
    lib.orc_bf16_value.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_round.restype = ctypes.c_uint16
    lib.orc_bf16_round.argtypes = [ctypes.c_double]
    lib.orc_e4m3_value.restype = ctypes.c_double
    lib.orc_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_encode.restype = ctypes.c_uint8
    lib.orc_e4m3_encode.argtypes = [ctypes.c_double]
    lib.orc_ue8m0_exponent.restype = _I
    lib.orc_ue8m0_exponent.argtypes = [ctypes.c_double]
    lib.orc_ue8m0_byte.restype = ctypes.c_uint8
    lib.orc_ue8m0_byte.argtypes = [ctypes.c_double]
    lib.orc_exponent_margin.restype = ctypes.c_double
    lib.orc_exponent_margin.argtypes = [ctypes.c_double]
    for name in ("orc_bf16_round_n", "orc_e4m3_encode_n", "orc_ue8m0_byte_n"):
        getattr(lib, name).restype = None
        getattr(lib, name).argtypes = [_P, _P, _I64]
    lib.orc_default_threads.restype = _I
    lib.orc_default_threads.argtypes = []
    lib.orc_qk_norm_rope.restype = _I
    lib.orc_qk_norm_rope.argtypes = [_P, _P, _I64, _I, _I, _I, _I, ctypes.c_float,
                                     _P, _P, _P, _I64, _I, _I, _P, _P, _P, _I]
    lib.orc_dsv4_gather.restype = _I
    lib.orc_dsv4_gather.argtypes = [_P, _I64, _I, _P, _I64, _P]
    lib.orc_dsv4.restype = _I
    lib.orc_dsv4.argtypes = [_P, _P, _P, _I64, _I, ctypes.c_float, _P, _P, _P, _I64,
                             _P, _P, _P, _I64, _I, _P, _P, _P, _P, _P, _I]
    return lib


_LIB = None


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = _declare(ctypes.CDLL(build()))
    return _LIB


def load_variant(path: str) -> ctypes.CDLL:
    """Load another build of oracle.c (used by the mutation tests)."""
    return _declare(ctypes.CDLL(path))


def unload_variant(handle: ctypes.CDLL) -> None:
    """dlclose a library returned by ``load_variant``."""
    import _ctypes
    _ctypes.dlclose(handle._handle)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _need(a, dtype, name):
    if not isinstance(a, np.ndarray) or a.dtype != dtype or not a.flags.c_contiguous:
        raise OracleError(f"{name}: need a C-contiguous numpy {np.dtype(dtype).name} array")
    return a


def bf16_round(values, _lib=None) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    (_lib or lib()).orc_bf16_round_n(_ptr(v), _ptr(out), v.size)
    return out


def e4m3_encode(values, _lib=None) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, np.uint8)
    (_lib or lib()).orc_e4m3_encode_n(_ptr(v), _ptr(out), v.size)
    return out


def ue8m0_byte(amax, _lib=None) -> np.ndarray:
    v = np.ascontiguousarray(amax, dtype=np.float64)
    out = np.empty(v.shape, np.uint8)
    (_lib or lib()).orc_ue8m0_byte_n(_ptr(v), _ptr(out), v.size)
    return out


def default_threads() -> int:
    return lib().orc_default_threads()


def qk_norm_rope(qkv, num_heads_q, num_heads_k, num_heads_v, head_dim, eps,
                 q_weight, k_weight, cos_sin, positions, is_neox=True, rot_dim=None,
                 want_ref=False, nthreads=0, out=None, _lib=None):
    """Packed-QKV per-head RMSNorm + RoPE.

    qkv: uint16 [T, (Hq+Hk+Hv)*D] (bf16 bits).  Returns ``(out, ref, mag)``: out
    is the full packed tensor (bf16 bits, V copied through), ref/mag are fp64
    [T, Hq+Hk, D] (None unless ``want_ref``).
    """
    L = _lib or lib()
    _need(qkv, np.uint16, "qkv")
    _need(q_weight, np.uint16, "q_weight")
    _need(k_weight, np.uint16, "k_weight")
    _need(cos_sin, np.float32, "cos_sin")
    _need(positions, np.int64, "positions")
    T = qkv.shape[0]
    NR = num_heads_q + num_heads_k
    rot = head_dim if rot_dim is None else rot_dim
    if cos_sin.shape[1] != rot:
        raise OracleError("cos_sin width must equal the rotary width")
    if out is None:
        out = np.empty_like(qkv)
    ref = np.empty((T, NR, head_dim), np.float64) if want_ref else None
    mag = np.empty((T, NR, head_dim), np.float64) if want_ref else None
    rc = L.orc_qk_norm_rope(_ptr(qkv), _ptr(out), T, num_heads_q, num_heads_k, num_heads_v,
                            head_dim, float(eps), _ptr(q_weight), _ptr(k_weight), _ptr(cos_sin),
                            cos_sin.shape[0], rot, 1 if is_neox else 0, _ptr(positions),
                            _ptr(ref), _ptr(mag), nthreads)
    if rc != 0:
        raise OracleError(f"orc_qk_norm_rope returned {rc}")
    return out, ref, mag


def dsv4(q, kv, eps, q_weight, kv_weight, cos_sin, positions, slot_mapping, kv_cache,
         want_ref=False, nthreads=0, q_out=None, _lib=None):
    """DSV4 Q norm+RoPE and KV norm+RoPE+quantise+insert.

    q: uint16 [T, H, 512]; kv: uint16 [T, 512]; kv_cache: uint8
    [num_blocks, block_size, 584], updated in place.  Returns a dict with
    ``q`` (bf16 bits) and, if ``want_ref``, fp64 ``q_ref``, ``q_mag``,
    ``kv_ref``, ``kv_mag`` and ``exp_margin`` [T, 7].
    """
    L = _lib or lib()
    _need(q, np.uint16, "q")
    _need(kv, np.uint16, "kv")
    _need(q_weight, np.uint16, "q_weight")
    _need(kv_weight, np.uint16, "kv_weight")
    _need(cos_sin, np.float32, "cos_sin")
    _need(positions, np.int64, "positions")
    _need(slot_mapping, np.int64, "slot_mapping")
    _need(kv_cache, np.uint8, "kv_cache")
    T, H = q.shape[0], q.shape[1]
    if q_out is None:
        q_out = np.empty_like(q)
    res = {"q": q_out}
    if want_ref:
        res["q_ref"] = np.empty(q.shape, np.float64)
        res["q_mag"] = np.empty(q.shape, np.float64)
        res["kv_ref"] = np.empty((T, DSV4_DIM), np.float64)
        res["kv_mag"] = np.empty((T, DSV4_DIM), np.float64)
        res["exp_margin"] = np.empty((T, DSV4_NBLOCK), np.float64)
    g = res.get
    rc = L.orc_dsv4(_ptr(q), _ptr(q_out), _ptr(kv), T, H, float(eps), _ptr(q_weight),
                    _ptr(kv_weight), _ptr(cos_sin), cos_sin.shape[0], _ptr(positions),
                    _ptr(slot_mapping), _ptr(kv_cache), kv_cache.shape[0], kv_cache.shape[1],
                    _ptr(g("q_ref")), _ptr(g("q_mag")), _ptr(g("kv_ref")), _ptr(g("kv_mag")),
                    _ptr(g("exp_margin")), nthreads)
    if rc != 0:
        raise OracleError(f"orc_dsv4 returned {rc}")
    return res


def dsv4_gather(kv_cache, slots, _lib=None):
    """bf16 bits [n, 512] read back from the entries at ``slots`` (see oracle.h)."""
    L = _lib or lib()
    _need(kv_cache, np.uint8, "kv_cache")
    _need(slots, np.int64, "slots")
    out = np.empty((slots.size, DSV4_DIM), np.uint16)
    rc = L.orc_dsv4_gather(_ptr(kv_cache), kv_cache.shape[0], kv_cache.shape[1], _ptr(slots),
                           slots.size, _ptr(out))
    if rc != 0:
        raise OracleError(f"orc_dsv4_gather returned {rc}")
    return out
