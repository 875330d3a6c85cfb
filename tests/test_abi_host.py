"""The C ABI on the host: symbols, status strings, validation, dispatch.

No call here reaches a kernel launch: every call either fails host-side
validation (the pointers passed are never dereferenced) or has nothing to do
(num_tokens == 0).  Runs without a GPU.
"""
import ctypes
import os
import re

import pytest

import kv_quant_cache_gb300 as kvq
from kv_quant_cache_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return kvq.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\(", text, flags=re.M)))


def test_header_declares_the_operators():
    names = declared_functions()
    for n in ("fused_qk_norm_rope", "dsv4_qnorm_rope_kv_rope_quant_insert", "kvq_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), f"libkvq.so does not export {name}"


def test_status_strings(L):
    for s in range(7):
        assert kvq.status_string(s)
    assert kvq.status_string(99) == "unknown kvq_status"


# fake, never-dereferenced device addresses for validation tests
A16 = 0x10000
MIS = 0x10008  # 8-byte but not 16-byte aligned


def _qk_invalid(qkv, T, hq, hk, hv, d, eps, qw, kw, cs, neox, pos, rot):
    """True when the documented validation rejects these arguments (or there
    is nothing to do), i.e. when the call cannot reach a kernel launch."""
    import math
    ptrs = (qkv, qw, kw, cs, pos)
    return (T <= 0 or min(hq, hk, hv) < 0 or hq + hk == 0 or d not in (64, 128, 256)
            or neox not in (0, 1) or rot < 16 or rot > d or rot % 16
            or not math.isfinite(eps) or eps < 0 or T * (hq + hk + 1) >= 2**31
            or any(p is None for p in ptrs)
            or any(p % a for p, a in zip(ptrs, (16, 16, 16, 16, 8))))


def qk(L, qkv=A16, T=4, hq=2, hk=1, hv=1, d=128, eps=1e-6, qw=A16, kw=A16, cs=A16, neox=1,
       pos=A16, rot=None):
    rot = d if rot is None else rot
    # fake addresses must never reach a launch
    assert _qk_invalid(qkv, T, hq, hk, hv, d, eps, qw, kw, cs, neox, pos, rot)
    return L.fused_qk_norm_rope_ex(qkv, T, hq, hk, hv, d, eps, qw, kw, cs, rot, neox, pos, None)


def dsv4(L, q=A16, kv=A16, T=4, H=2, eps=1e-6, qw=A16, kvw=A16, cs=A16, pos=A16, slot=A16,
         cache=A16, bs=64):
    import math
    ptrs = (q, kv, qw, kvw, cs, pos, slot, cache)
    invalid = (T <= 0 or H < 1 or bs < 1 or T * (H + 1) >= 2**31 or not math.isfinite(eps)
               or eps < 0 or any(p is None for p in ptrs)
               or any(p % a for p, a in zip(ptrs, (16, 16, 16, 16, 16, 8, 8, 8))))
    assert invalid  # fake addresses must never reach a launch
    return L.dsv4_qnorm_rope_kv_rope_quant_insert(q, kv, T, H, eps, qw, kvw, cs, pos, slot, cache,
                                                  bs, None)


def test_qk_validation(L):
    assert qk(L, qkv=None) == kvq.KVQ_ERR_NULL
    assert qk(L, pos=None) == kvq.KVQ_ERR_NULL
    assert qk(L, T=-1) == kvq.KVQ_ERR_SHAPE
    assert qk(L, hq=-1) == kvq.KVQ_ERR_SHAPE
    assert qk(L, d=96) == kvq.KVQ_ERR_UNSUPPORTED
    assert qk(L, d=512) == kvq.KVQ_ERR_UNSUPPORTED
    assert qk(L, neox=2) == kvq.KVQ_ERR_UNSUPPORTED
    assert qk(L, rot=8) == kvq.KVQ_ERR_UNSUPPORTED
    assert qk(L, rot=24) == kvq.KVQ_ERR_UNSUPPORTED
    assert qk(L, d=64, rot=128) == kvq.KVQ_ERR_UNSUPPORTED
    assert qk(L, rot=0) == kvq.KVQ_ERR_UNSUPPORTED
    # the plain entry point validates the same way (rotary_dim = head_dim)
    assert L.fused_qk_norm_rope(A16, 4, 2, 1, 1, 96, 1e-6, A16, A16, A16, 1, A16,
                                None) == kvq.KVQ_ERR_UNSUPPORTED
    assert L.fused_qk_norm_rope(A16, 4, 2, 1, 1, 128, 1e-6, A16, A16, A16, 3, A16,
                                None) == kvq.KVQ_ERR_UNSUPPORTED
    assert qk(L, eps=-1.0) == kvq.KVQ_ERR_VALUE
    assert qk(L, eps=float("nan")) == kvq.KVQ_ERR_VALUE
    assert qk(L, eps=float("inf")) == kvq.KVQ_ERR_VALUE
    assert qk(L, qkv=MIS) == kvq.KVQ_ERR_ALIGN
    assert qk(L, cs=MIS) == kvq.KVQ_ERR_ALIGN
    assert qk(L, pos=A16 + 4) == kvq.KVQ_ERR_ALIGN
    assert qk(L, T=1 << 30, hq=2, hk=0) == kvq.KVQ_ERR_SHAPE   # index range
    # sums and products that overflow 32 or 64 bits are rejected, not wrapped
    INT_MAX = 2**31 - 1
    assert qk(L, hq=INT_MAX, hk=INT_MAX, hv=0) == kvq.KVQ_ERR_SHAPE
    assert qk(L, hq=INT_MAX, hk=1, hv=INT_MAX) == kvq.KVQ_ERR_SHAPE
    assert qk(L, T=2**62, hq=4, hk=0) == kvq.KVQ_ERR_SHAPE
    assert qk(L, T=2**63 - 1, hq=1, hk=0, hv=0) == kvq.KVQ_ERR_SHAPE
    # nothing to do: OK without a launch, even with NULL pointers
    assert qk(L, qkv=None, qw=None, kw=None, cs=None, pos=None, T=0) == kvq.KVQ_OK
    assert qk(L, qkv=None, qw=None, kw=None, cs=None, pos=None, hq=0, hk=0) == kvq.KVQ_OK
    # valid layouts still reach the pointer checks (and stop there)
    for d, rot, neox in ((64, 64, 0), (256, 128, 1), (128, 32, 0), (64, 16, 1)):
        assert qk(L, d=d, rot=rot, neox=neox, qkv=None) == kvq.KVQ_ERR_NULL
        assert qk(L, d=d, rot=rot, neox=neox, qkv=MIS) == kvq.KVQ_ERR_ALIGN


def test_dsv4_validation(L):
    assert dsv4(L, q=None) == kvq.KVQ_ERR_NULL
    assert dsv4(L, slot=None) == kvq.KVQ_ERR_NULL
    assert dsv4(L, cache=None) == kvq.KVQ_ERR_NULL
    assert dsv4(L, T=-3) == kvq.KVQ_ERR_SHAPE
    assert dsv4(L, H=0) == kvq.KVQ_ERR_SHAPE
    assert dsv4(L, bs=0) == kvq.KVQ_ERR_SHAPE
    assert dsv4(L, T=1 << 24, H=128) == kvq.KVQ_ERR_SHAPE
    assert dsv4(L, T=1, H=2**31 - 1) == kvq.KVQ_ERR_SHAPE
    assert dsv4(L, T=2**62, H=3) == kvq.KVQ_ERR_SHAPE
    assert L.kvq_dsv4_dispatch_path(2**62, 3) == 1
    assert L.kvq_dsv4_dispatch_path(1, 2**31 - 1) == 1
    assert L.kvq_qk_config_for(2**62, 3, 1) == L.kvq_qk_config_for(1 << 20, 32, 8)
    assert dsv4(L, eps=float("nan")) == kvq.KVQ_ERR_VALUE
    assert dsv4(L, q=MIS) == kvq.KVQ_ERR_ALIGN
    assert dsv4(L, kv=MIS) == kvq.KVQ_ERR_ALIGN
    assert dsv4(L, qw=MIS) == kvq.KVQ_ERR_ALIGN
    assert dsv4(L, cache=A16 + 4) == kvq.KVQ_ERR_ALIGN
    assert dsv4(L, q=None, kv=None, qw=None, kvw=None, cs=None, pos=None, slot=None, cache=None,
                T=0) == kvq.KVQ_OK


def test_cache_alignment_rule_is_eight_bytes(L):
    # an 8-byte aligned cache passes alignment; make another argument invalid so
    # that nothing launches, and check that the reported error is not ALIGN.
    assert dsv4(L, cache=A16 + 8, bs=0) == kvq.KVQ_ERR_SHAPE
    assert dsv4(L, cache=A16 + 8, slot=None) == kvq.KVQ_ERR_NULL


def test_dispatch_threshold(L):
    old = kvq.set_dsv4_dispatch_threshold(-1)
    try:
        default = kvq.dsv4_dispatch_threshold()
        assert default > 0
        assert kvq.dsv4_dispatch_path(1, 128) == 0
        assert kvq.dsv4_dispatch_path(131072, 128) == 1
        kvq.set_dsv4_dispatch_threshold(0)
        assert kvq.dsv4_dispatch_path(1, 1) == 1
        kvq.set_dsv4_dispatch_threshold(1 << 40)
        assert kvq.dsv4_dispatch_path(131072, 128) == 0
        assert kvq.set_dsv4_dispatch_threshold(-1) == 1 << 40
        assert kvq.dsv4_dispatch_threshold() == default
        # the boundary is a program count T * (H + 1)
        kvq.set_dsv4_dispatch_threshold(129 * 4)
        assert kvq.dsv4_dispatch_path(3, 128) == 0 and kvq.dsv4_dispatch_path(4, 128) == 1
    finally:
        kvq.set_dsv4_dispatch_threshold(old)


@pytest.mark.parametrize("value,expected", [("1234", 1234), ("0", 0), ("abc", 65536),
                                            ("-5", 65536), ("12x", 65536), ("", 65536)])
def test_dispatch_threshold_from_environment(L, value, expected):
    """KVQ_DSV4_DISPATCH_THRESHOLD is read once, in a fresh process; anything
    but a plain non-negative integer leaves the built-in default."""
    import subprocess
    import sys
    env = dict(os.environ, KVQ_DSV4_DISPATCH_THRESHOLD=value)
    code = ("import ctypes, sys; L = ctypes.CDLL(sys.argv[1]); "
            "L.kvq_dsv4_dispatch_threshold.restype = ctypes.c_int64; "
            "print(L.kvq_dsv4_dispatch_threshold())")
    out = subprocess.run([sys.executable, "-c", code, kvq.LIB_PATH], env=env, check=True,
                         capture_output=True, text=True).stdout
    assert int(out) == expected


def test_binding_rejects_cpu_tensors(L):
    import torch
    x = torch.zeros(2, 4 * 128, dtype=torch.bfloat16)
    w = torch.zeros(128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        kvq.fused_qk_norm_rope(x, 2, 1, 1, 128, 1e-6, w, w, torch.zeros(4, 128), True,
                               torch.zeros(2, dtype=torch.int64))


def test_binding_rejects_short_operands(L):
    """Sizes the C ABI cannot see (weights, tables, per-token arrays) are
    checked by the binding before anything reaches the library."""
    import torch
    bf, i64 = torch.bfloat16, torch.int64
    x = torch.zeros(2, 4 * 128, dtype=bf)
    w = torch.zeros(128, dtype=bf)
    cs = torch.zeros(4, 128)
    pos = torch.zeros(2, dtype=i64)
    with pytest.raises(ValueError, match="head_dim values"):
        kvq.fused_qk_norm_rope(x, 2, 1, 1, 128, 1e-6, w[:64], w, cs, True, pos)
    with pytest.raises(ValueError, match="one value per token"):
        kvq.fused_qk_norm_rope(x, 2, 1, 1, 128, 1e-6, w, w, cs, True, pos[:1])
    q = torch.zeros(2, 3, 512, dtype=bf)
    kv = torch.zeros(2, 512, dtype=bf)
    w5 = torch.zeros(512, dtype=bf)
    cs5 = torch.zeros(8, 64)
    cache = torch.zeros(1, 64, 584, dtype=torch.uint8)
    with pytest.raises(ValueError, match="512 values"):
        kvq.dsv4_qnorm_rope_kv_rope_quant_insert(q, kv, 1e-6, w5[:256], w5, cs5, pos, pos, cache)
    with pytest.raises(ValueError, match=r"\[max_pos, 64\]"):
        kvq.dsv4_qnorm_rope_kv_rope_quant_insert(q, kv, 1e-6, w5, w5, cs5[:, :32], pos, pos,
                                                 cache)
    with pytest.raises(ValueError, match="one value per token"):
        kvq.dsv4_qnorm_rope_kv_rope_quant_insert(q, kv, 1e-6, w5, w5, cs5, pos, pos[:1], cache)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(kvq, "_LIB", None)
    monkeypatch.setattr(kvq, "LIB_PATH", str(tmp_path / "libkvq.so"))
    with pytest.raises(kvq.KvqError):
        kvq.lib()


def test_launch_config_table(L):
    for op in ("qk", "dsv4"):
        names = kvq.configs(op)
        assert len(names) >= 2 and len(set(names)) == len(names)
        assert getattr(L, f"kvq_{op}_config_name")(len(names)) is None
        assert getattr(L, f"kvq_{op}_config_name")(-1) is None
        prev = kvq.set_config(op, len(names) - 1)
        try:
            assert kvq.set_config(op, 0) == len(names) - 1
            with pytest.raises(ValueError):
                kvq.set_config(op, len(names))
            assert kvq.set_config(op, 0) == 0   # unchanged by the rejected id
        finally:
            kvq.set_config(op, prev)
    kvq.set_config("dsv4", 3)
    try:
        assert kvq.dsv4_config_for(131072, 128) == 3 and kvq.dsv4_config_for(1, 1) == 3
    finally:
        kvq.set_config("dsv4", -1)
    assert kvq.dsv4_config_for(1, 1) in range(len(kvq.configs("dsv4")))
    # automatic DSV4 shapes: the one-row grid below the threshold, the
    # persistent grid taking adjacent row pairs above it
    ds = kvq.configs("dsv4")
    assert ds[kvq.dsv4_config_for(16, 64)] == "tiles<4w,1row>"
    assert ds[kvq.dsv4_config_for(32768, 64)] == "stream<8w,85reg,pairs>"
    assert kvq.qk_config_for(32768, 32, 8) in range(len(kvq.configs("qk")))
    qk = kvq.configs("qk")
    # automatic QK shapes at head_dim 128: < 1216 Q+K rows small-batch,
    # < 128 MiB of Q+K rows (2^19 rows) register-pipelined, then TMA-staged
    assert qk[kvq.qk_config_for(17, 16, 8)] == "tiles<4w,1step>"
    assert qk[kvq.qk_config_for(30, 32, 8)] == "tiles<4w,1step>"   # 1200 rows
    assert qk[kvq.qk_config_for(31, 32, 8)] == "tiles<4w,4step>"   # 1240 rows
    assert qk[kvq.qk_config_for(5734, 32, 8)] == "tiles<4w,4step>"    # 229360 rows < 56 MiB
    assert qk[kvq.qk_config_for(5735, 32, 8)] == "bulk<24w,2st,3KB>"  # 229400 rows
    assert qk[kvq.qk_config_for(13107, 32, 8)] == "bulk<24w,2st,3KB>"  # 524280 rows < 128 MiB
    assert qk[kvq.qk_config_for(13108, 32, 8)] == "bulk<16w,2st,6KB>"
    assert qk[kvq.qk_config_for(32768, 32, 8)] == "bulk<16w,2st,6KB>"


def test_gather_validation(L):
    def g(cache=A16, bs=64, slots=A16, n=4, out=A16):
        ptrs = (cache, slots, out)
        assert (n <= 0 or bs < 1 or any(p is None for p in ptrs)
                or any(p % a for p, a in zip(ptrs, (8, 8, 16))))  # never a launch
        return L.dsv4_kv_cache_gather(cache, bs, slots, n, out, None)
    assert g(cache=None) == kvq.KVQ_ERR_NULL
    assert g(out=None) == kvq.KVQ_ERR_NULL
    assert g(n=-1) == kvq.KVQ_ERR_SHAPE
    assert g(bs=0) == kvq.KVQ_ERR_SHAPE
    assert g(cache=A16 + 4) == kvq.KVQ_ERR_ALIGN
    assert g(out=A16 + 8) == kvq.KVQ_ERR_ALIGN
    assert g(slots=A16 + 4) == kvq.KVQ_ERR_ALIGN
    assert g(cache=None, slots=None, out=None, n=0) == kvq.KVQ_OK


def test_out_of_place_validation(L):
    def o(q=A16, q_out=A16 + 2**20, kv=A16, T=4, H=2, eps=1e-6):
        qbytes = T * H * 1024
        overlap = q is not None and q_out is not None and q != q_out and \
            q < q_out + qbytes and q_out < q + qbytes
        assert (q is None or q_out is None or q_out % 16 or overlap or T <= 0)  # no launch
        return L.dsv4_qnorm_rope_kv_rope_quant_insert_out(q, q_out, kv, T, H, eps, A16, A16, A16,
                                                          A16, A16, A16, 64, None)
    assert o(q_out=None) == kvq.KVQ_ERR_NULL
    assert o(q_out=A16 + 2**20 + 8) == kvq.KVQ_ERR_ALIGN
    assert o(q_out=A16 + 1024) == kvq.KVQ_ERR_VALUE          # partial overlap
    assert o(q_out=A16 - 4096) == kvq.KVQ_ERR_VALUE
    assert o(T=0, q=None, q_out=None) == kvq.KVQ_OK


def test_checked_entry_points_validation(L):
    # every call below fails validation before any launch (fake addresses)
    E = A16 + 2**20
    args_qk = (A16, 4, 2, 1, 1, 128, 1e-6, A16, A16, A16)
    assert L.fused_qk_norm_rope_checked(*args_qk, 64, 128, 1, A16, None, None) == kvq.KVQ_ERR_NULL
    assert L.fused_qk_norm_rope_checked(*args_qk, 64, 128, 1, A16, E + 2, None) == kvq.KVQ_ERR_ALIGN
    assert L.fused_qk_norm_rope_checked(*args_qk, -1, 128, 1, A16, E, None) == kvq.KVQ_ERR_SHAPE
    assert L.fused_qk_norm_rope_checked(A16, 4, 2, 1, 1, 96, 1e-6, A16, A16, A16, 64, 96, 1, A16,
                                        E, None) == kvq.KVQ_ERR_UNSUPPORTED
    head = (A16, A16, A16, 4, 2, 1e-6, A16, A16, A16)
    assert L.dsv4_qnorm_rope_kv_rope_quant_insert_checked(
        *head, 64, A16, A16, A16, 8, 64, None, None) == kvq.KVQ_ERR_NULL
    assert L.dsv4_qnorm_rope_kv_rope_quant_insert_checked(
        *head, 64, A16, A16, A16, -1, 64, E, None) == kvq.KVQ_ERR_SHAPE
    assert L.dsv4_qnorm_rope_kv_rope_quant_insert_checked(
        *head, -5, A16, A16, A16, 8, 64, E, None) == kvq.KVQ_ERR_SHAPE
    assert L.dsv4_qnorm_rope_kv_rope_quant_insert_checked(
        *head, 64, A16, A16, A16, 8, 64, E + 1, None) == kvq.KVQ_ERR_ALIGN
    assert L.dsv4_kv_cache_gather_checked(A16, 8, 64, A16, 4, A16, None, None) == kvq.KVQ_ERR_NULL
    assert L.dsv4_kv_cache_gather_checked(A16, -1, 64, A16, 4, A16, E, None) == kvq.KVQ_ERR_SHAPE
    assert L.dsv4_kv_cache_gather_checked(A16, 8, 64, A16, 4, A16 + 8, E, None) == kvq.KVQ_ERR_ALIGN


def test_stage_wait_limit_round_trip(L):
    """The staged shapes' wait limit: returns the previous value, default 2^22."""
    old = kvq.set_stage_wait_limit(17)
    try:
        assert old == 1 << 22
        assert kvq.set_stage_wait_limit(0) == 17
        assert kvq.set_stage_wait_limit(5) == 0
    finally:
        assert kvq.set_stage_wait_limit(old) == 5


def test_programmatic_launch_switch(L):
    old = kvq.set_programmatic_launch(False)
    try:
        assert old is True   # on by default
        assert kvq.set_programmatic_launch(True) is False
        assert kvq.set_programmatic_launch(False) is True
    finally:
        kvq.set_programmatic_launch(old)


def test_stage_events_rejects_null(L):
    """The staging-event read-out checks its pointers before touching the
    device."""
    x = ctypes.c_uint64(0)
    assert L.kvq_stage_events(None, ctypes.addressof(x), 0) == kvq.KVQ_ERR_NULL
    assert L.kvq_stage_events(ctypes.addressof(x), None, 1) == kvq.KVQ_ERR_NULL


class _FakeTensor:
    """Stands in for a tensor in the binding's device check (no GPU here)."""

    def __init__(self, device):
        self.is_cuda = device >= 0
        self._device = device

    def get_device(self):
        return self._device


def test_binding_device_check():
    """Every CUDA tensor of one call must be on one device; pinned host
    tensors (get_device() == -1) may take part on any; the call runs on the
    tensors' device."""
    F = _FakeTensor
    assert kvq._device(F(1), F(1), None, F(-1)) == 1
    assert kvq._device(F(-1), F(-1)) == -1
    assert kvq._device(F(-1), F(3)) == 3
    with pytest.raises(ValueError, match="same device"):
        kvq._device(F(0), F(-1), F(1))
