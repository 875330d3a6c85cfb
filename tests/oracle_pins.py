"""Pins of the CPU oracle to things other than itself.

Each ``pin_*`` function takes a loaded oracle library (``oracle.lib()`` or a
deliberately broken variant built by the mutation test) and raises
AssertionError when the oracle disagrees with an independent fact:

* torch's CPU casts to ``bfloat16`` and ``float8_e4m3fn`` (library routines);
* ``torch.nn.functional.rms_norm`` in fp64 (library routine);
* rotation written as complex multiplication with numpy (a different
  formulation of the same rotation);
* exact rational arithmetic (``fractions.Fraction``) for the UE8M0 exponent;
* closed forms and hand-derived cache entries.

None of these re-types the oracle's own formulas.
"""
from __future__ import annotations

import bisect
import functools
import math
from fractions import Fraction

import numpy as np
import torch

import oracle
import workloads as wl

EPS = 1e-6


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def _bf16_value(bits: np.ndarray) -> np.ndarray:
    """bf16 bits -> float64 through the binary32 bit layout (numpy view)."""
    with np.errstate(invalid="ignore"):
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _to_bits(values) -> np.ndarray:
    return wl.bf16_bits(torch.as_tensor(np.asarray(values, np.float32)).to(torch.bfloat16))


def _is_nearest_bf16(bits: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """True where ``bits`` is the round-to-nearest-even bf16 of the exact ``ref``."""
    bits = bits.astype(np.int64).ravel()
    ref = ref.ravel()
    sign = bits & 0x8000
    mag = bits & 0x7FFF
    v = _bf16_value(bits.astype(np.uint16))
    up = _bf16_value((sign | np.minimum(mag + 1, 0x7F80)).astype(np.uint16))
    dn = _bf16_value((sign | np.maximum(mag - 1, 0)).astype(np.uint16))
    d = np.abs(ref - v)
    du = np.abs(ref - up)
    dd = np.where(mag > 0, np.abs(ref - dn), np.inf)
    same_sign = (ref == 0) | ((ref < 0) == (sign != 0)) | (mag == 0)
    ok = (d <= du) & (d <= dd) & same_sign
    tie = ((d == du) | (d == dd)) & (d > 0)
    return ok & (~tie | (mag % 2 == 0))


def _qk_inputs(T, Hq, Hk, Hv, D=128, seed=3, max_pos=64, positions=None, theta=1e4):
    d = wl.make_qk(T, Hq, Hk, Hv, D, theta, max_pos, "uniform", seed)
    pos = wl.host(d["positions"]) if positions is None else np.asarray(positions, np.int64)
    return dict(qkv=wl.bf16_bits(d["qkv"]), q_weight=wl.bf16_bits(d["q_weight"]),
                k_weight=wl.bf16_bits(d["k_weight"]), cos_sin=wl.host(d["cos_sin"]),
                positions=np.ascontiguousarray(pos))


def _run_qk(L, inp, Hq, Hk, Hv, D=128, is_neox=True, eps=EPS, nthreads=1):
    return oracle.qk_norm_rope(inp["qkv"], Hq, Hk, Hv, D, eps, inp["q_weight"],
                               inp["k_weight"], inp["cos_sin"], inp["positions"],
                               is_neox=is_neox, want_ref=True, nthreads=nthreads, _lib=L)


def _dsv4_inputs(T, H, seed=11, max_pos=64, num_blocks=8, block_size=4, slots="distinct"):
    d = wl.make_dsv4(T, H, 1e4, max_pos, num_blocks, block_size, slots, seed)
    return dict(q=wl.bf16_bits(d["q"]), kv=wl.bf16_bits(d["kv"]),
                q_weight=wl.bf16_bits(d["q_weight"]), kv_weight=wl.bf16_bits(d["kv_weight"]),
                cos_sin=wl.host(d["cos_sin"]), positions=wl.host(d["positions"]),
                slot_mapping=wl.host(d["slot_mapping"]), kv_cache=wl.host(d["kv_cache"]))


def _run_dsv4(L, inp, eps=EPS, nthreads=1, want_ref=True):
    cache = inp["kv_cache"].copy()
    res = oracle.dsv4(inp["q"], inp["kv"], eps, inp["q_weight"], inp["kv_weight"],
                      inp["cos_sin"], inp["positions"], inp["slot_mapping"], cache,
                      want_ref=want_ref, nthreads=nthreads, _lib=L)
    res["cache"] = cache
    return res


def brute_ue8m0_exponent(amax: float) -> int:
    """Smallest integer e with 448 * 2^e >= amax, in exact rational arithmetic."""
    A = Fraction(amax)
    lo, hi = -400, 400  # predicate false at lo, true at hi for any positive double
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if Fraction(448) * (Fraction(2) ** mid) >= A:
            hi = mid
        else:
            lo = mid
    return hi


@functools.lru_cache(maxsize=1)
def _e4m3_positive_values():
    """Exact values of the finite non-negative e4m3fn codes 0..126, decoded by
    torch's float8_e4m3fn (increasing with the code)."""
    codes = np.arange(127, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return [Fraction(float(v)) for v in vals]


def brute_e4m3_code(v: float) -> int:
    """The e4m3fn code nearest to the exact value ``v`` (|v| <= 448), ties to
    the even code, sign kept: a search over the decoded code values in exact
    rational arithmetic."""
    tab = _e4m3_positive_values()
    a = abs(Fraction(v))
    assert a <= 448
    i = bisect.bisect_left(tab, a)
    cands = [c for c in (i - 1, i) if 0 <= c < len(tab)]
    best = min(cands, key=lambda c: (abs(tab[c] - a), c & 1))
    return (0x80 if math.copysign(1.0, v) < 0 else 0) | best


def brute_exponent_margin(amax: float) -> float:
    """|amax - B| / amax for the nearer of the boundaries B = 448 * 2^(e-1),
    448 * 2^e around amax's exponent decision e, in exact arithmetic."""
    if amax <= 0:
        return math.inf
    A = Fraction(amax)
    e = brute_ue8m0_exponent(amax)
    hi = Fraction(448) * Fraction(2) ** e
    lo = hi / 2
    assert lo < A <= hi
    return float(min((hi - A) / A, (A - lo) / A))


# ---------------------------------------------------------------------------
# scalar codecs
# ---------------------------------------------------------------------------

def pin_bf16_value_and_roundtrip(L):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = np.array([L.orc_bf16_value(int(b)) for b in bits])
    want = _bf16_value(bits)
    fin = np.isfinite(want)
    assert np.array_equal(vals[fin], want[fin])
    back = oracle.bf16_round(want[fin], _lib=L)
    assert np.array_equal(back, bits[fin]), "bf16 round trip"


def pin_bf16_vs_torch(L):
    rng = np.random.default_rng(7)
    raw = rng.integers(0, 2**32, 300_000, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 2**16, 50_000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    near = np.concatenate([ties + 1, ties - 1])
    f = np.concatenate([raw, ties, near]).view(np.float32)
    f = f[np.isfinite(f)]
    want = wl.bf16_bits(torch.from_numpy(f).to(torch.bfloat16))
    got = oracle.bf16_round(f.astype(np.float64), _lib=L)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"bf16 vs torch: {bad.size} mismatches, first {f[bad[:3]]}"


def pin_bf16_single_rounding(L):
    # 1 + 2^-8 + 2^-40 is just above the midpoint between 1 and 1 + 2^-7: one
    # rounding step gives 1 + 2^-7 (0x3f81); a detour through fp32 would lose
    # the 2^-40 and then round the exact tie to even (0x3f80).
    assert L.orc_bf16_round(1.0 + 2.0**-8 + 2.0**-40) == 0x3F81
    assert L.orc_bf16_round(1.0 + 2.0**-8) == 0x3F80            # tie -> even
    assert L.orc_bf16_round(1.0 + 3 * 2.0**-8) == 0x3F82        # tie -> even (up)
    assert L.orc_bf16_round(-(1.0 + 2.0**-8 + 2.0**-40)) == 0xBF81
    assert L.orc_bf16_round(2.0**-133) == 0x0001                # smallest subnormal
    assert L.orc_bf16_round(2.0**-134) == 0x0000                # tie with 0 -> even
    assert L.orc_bf16_round(-0.0) == 0x8000


def pin_e4m3_decode_vs_torch(L):
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([L.orc_e4m3_value(int(c)) for c in codes])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0**-9


def pin_e4m3_roundtrip(L):
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = np.array([L.orc_e4m3_value(int(c)) for c in codes])
    vals[codes == 0x80] = -0.0
    assert np.array_equal(oracle.e4m3_encode(vals, _lib=L), codes)
    # one rounding from fp64: 2^-40 above the midpoint of 1.125 and 1.25 rounds
    # up, 2^-40 below it down; the exact midpoints tie to the even code
    assert L.orc_e4m3_encode(1.1875 + 2.0**-40) == 0x3A
    assert L.orc_e4m3_encode(1.1875 - 2.0**-40) == 0x39
    assert L.orc_e4m3_encode(1.1875) == 0x3A and L.orc_e4m3_encode(1.0625) == 0x38
    for v in (1.1875 + 2.0**-40, 1.1875 - 2.0**-40, -(1.0625 + 2.0**-41), 3.0 * 2.0**-10):
        assert L.orc_e4m3_encode(v) == brute_e4m3_code(v), v


def pin_e4m3_vs_torch(L):
    rng = np.random.default_rng(8)
    n = 400_000
    mags = np.exp2(rng.uniform(-13, np.log2(448.0), n))
    sgn = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    pos_vals = np.array([L.orc_e4m3_value(c) for c in range(127)])
    mids = (pos_vals[:-1] + pos_vals[1:]) / 2  # exact ties
    m32 = mids.astype(np.float32)
    near = np.concatenate([np.nextafter(m32, np.float32(0)), np.nextafter(m32, np.float32(1e9))])
    f = np.concatenate([(mags * sgn).astype(np.float32), m32, -m32, near, -near,
                        pos_vals.astype(np.float32)])
    want = torch.from_numpy(f).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(f.astype(np.float64), _lib=L)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"e4m3 vs torch: {bad.size} mismatches, first {f[bad[:3]]}"


def pin_ue8m0_hand(L):
    cases = {
        448.0: 0,                      # exactly representable: 2^0
        float(np.nextafter(448.0, 1e9)): 1,
        1.0: -8,                       # 448 / 256 = 1.75 >= 1 > 0.875
        3.5: -7,                       # 448 * 2^-7 = 3.5 exactly
        float(np.nextafter(3.5, 9.0)): -6,
        1.75: -8,
        0.875: -9,
    }
    for amax, e in cases.items():
        assert L.orc_ue8m0_exponent(amax) == e, amax
        assert L.orc_ue8m0_byte(amax) == e + 127, amax
    assert L.orc_ue8m0_byte(0.0) == 0
    assert L.orc_ue8m0_byte(1e-40) == 0                  # e = -141, clamped
    assert L.orc_ue8m0_byte(448.0 * 2.0**127) == 254
    assert L.orc_ue8m0_byte(448.0 * 2.0**200) == 254     # clamped


def pin_ue8m0_bruteforce(L):
    rng = np.random.default_rng(9)
    raw = rng.integers(0x00800000, 0x7F000000, 3000, dtype=np.uint64).astype(np.uint32)
    vals = [float(v) for v in raw.view(np.float32)]
    for k in range(-130, 121, 7):   # boundaries 448 * 2^k and their fp32 neighbours
        b = np.float32(448.0 * 2.0**k)
        vals += [float(b), float(np.nextafter(b, np.float32(0))), float(np.nextafter(b, np.float32(3e38)))]
    got = oracle.ue8m0_byte(np.array(vals), _lib=L)
    for v, g in zip(vals, got):
        e = brute_ue8m0_exponent(v)
        assert int(g) == min(max(e + 127, 0), 254), (v, int(g), e)


# ---------------------------------------------------------------------------
# packed-QKV operator
# ---------------------------------------------------------------------------

def _textbook(x_bits, w_bits, D, eps=EPS):
    x = torch.from_numpy(_bf16_value(x_bits).reshape(-1, D))
    w = torch.from_numpy(_bf16_value(w_bits))
    return torch.nn.functional.rms_norm(x, (D,), weight=w, eps=eps).numpy()


def pin_qk_textbook_rmsnorm(L):
    T, Hq, Hk, Hv, D = 3, 3, 2, 1, 128
    inp = _qk_inputs(T, Hq, Hk, Hv, D, positions=[0, 0, 0])
    out, ref, mag = _run_qk(L, inp, Hq, Hk, Hv, D)
    x = inp["qkv"].reshape(T, Hq + Hk + Hv, D)
    want_q = _textbook(x[:, :Hq].copy(), inp["q_weight"], D).reshape(T, Hq, D)
    want_k = _textbook(x[:, Hq:Hq + Hk].copy(), inp["k_weight"], D).reshape(T, Hk, D)
    np.testing.assert_allclose(ref[:, :Hq], want_q, rtol=1e-12, atol=0)
    np.testing.assert_allclose(ref[:, Hq:], want_k, rtol=1e-12, atol=0)
    qk_bits = out.reshape(T, Hq + Hk + Hv, D)[:, :Hq + Hk]
    assert _is_nearest_bf16(qk_bits, ref).all(), "outputs are the nearest bf16 of ref"
    # with unit weights the normalised row has mean square ms / (ms + eps)
    ones = _to_bits(np.ones(D))
    inp1 = dict(inp, q_weight=ones, k_weight=ones)
    _, ref1, _ = _run_qk(L, inp1, Hq, Hk, Hv, D)
    xs = _bf16_value(x[:, :Hq + Hk].copy())
    ms = (xs * xs).mean(-1)
    np.testing.assert_allclose((ref1 * ref1).mean(-1), ms / (ms + np.float32(EPS)), rtol=1e-12)


def pin_qk_all_equal_row(L):
    D = 128
    a = 0.375
    qkv = np.ascontiguousarray(np.tile(_to_bits(np.full(D, a)), (1, 2)))  # 1 Q + 1 K head
    w = _to_bits(np.full(D, 1.5))
    cs = np.zeros((1, D), np.float32)
    cs[0, :D // 2] = 1.0
    inp = dict(qkv=qkv, q_weight=w, k_weight=w, cos_sin=cs, positions=np.zeros(1, np.int64))
    _, ref, _ = _run_qk(L, inp, 1, 1, 0, D)
    eps = float(np.float32(EPS))
    np.testing.assert_allclose(ref, a / np.sqrt(a * a + eps) * 1.5, rtol=1e-14)


def _complex_rotate(n, cs_rows, neox, off, rot):
    half = rot // 2
    c = cs_rows[..., :half].astype(np.float64)
    s = cs_rows[..., half:rot].astype(np.float64)
    part = n[..., off:off + rot]
    if neox:
        z = part[..., :half] + 1j * part[..., half:]
    else:
        z = part[..., 0::2] + 1j * part[..., 1::2]
    zr = z * (c + 1j * s)
    out = n.copy()
    if neox:
        out[..., off:off + half] = zr.real
        out[..., off + half:off + rot] = zr.imag
    else:
        out[..., off:off + rot:2] = zr.real
        out[..., off + 1:off + rot:2] = zr.imag
    return out


def pin_qk_rope_complex(L):
    T, Hq, Hk, Hv, D = 4, 2, 2, 2, 128
    base = _qk_inputs(T, Hq, Hk, Hv, D, max_pos=4096, positions=[0, 0, 0, 0])
    _, n0, _ = _run_qk(L, base, Hq, Hk, Hv, D)
    pos = np.array([1, 17, 1000, 4095], np.int64)
    _, nr, mag = _run_qk(L, dict(base, positions=pos), Hq, Hk, Hv, D)
    want = _complex_rotate(n0, base["cos_sin"][pos][:, None, :], True, 0, D)
    assert np.all(np.abs(nr - want) <= 1e-14 * mag + 1e-300)
    # rotation keeps each pair's norm up to the table's own c^2 + s^2
    c = base["cos_sin"][pos][:, None, :D // 2].astype(np.float64)
    s = base["cos_sin"][pos][:, None, D // 2:].astype(np.float64)
    lhs = nr[..., :D // 2] ** 2 + nr[..., D // 2:] ** 2
    rhs = (n0[..., :D // 2] ** 2 + n0[..., D // 2:] ** 2) * (c * c + s * s)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12)


def pin_qk_rope_partial(L):
    """Partial and full rotation at head_dim 64 and 256, NeoX and interleaved pairs
    [IO1019 "Summary": the API carries is_neox; rotary_dim < head_dim rotates
    the leading dims]: the first rotary_dim dims of each head equal complex
    multiplication of their pairs by the table row (width rotary_dim), and
    every dim from rotary_dim on keeps its unrotated normalised value."""
    T, Hq, Hk, Hv = 3, 2, 1, 1
    pos = np.array([1, 700, 2000], np.int64)
    for D in (64, 256):
        for rot in (16, D // 2, D):
            for neox in (True, False):
                d = wl.make_qk(T, Hq, Hk, Hv, D, 1e4, 4096, "uniform", 7 + D + rot,
                               rotary_dim=rot)
                base = dict(qkv=wl.bf16_bits(d["qkv"]), q_weight=wl.bf16_bits(d["q_weight"]),
                            k_weight=wl.bf16_bits(d["k_weight"]), cos_sin=wl.host(d["cos_sin"]))

                def run(positions):
                    return oracle.qk_norm_rope(base["qkv"], Hq, Hk, Hv, D, EPS, base["q_weight"],
                                               base["k_weight"], base["cos_sin"], positions,
                                               is_neox=neox, rot_dim=rot, want_ref=True,
                                               nthreads=1, _lib=L)
                _, n0, _ = run(np.zeros(T, np.int64))          # position 0: no rotation
                _, nr, mag = run(pos)
                want = _complex_rotate(n0, base["cos_sin"][pos][:, None, :], neox, 0, rot)
                assert np.all(np.abs(nr - want) <= 1e-14 * mag + 1e-300), (D, rot, neox)
                assert np.array_equal(nr[..., rot:], n0[..., rot:]), (D, rot, neox)
                assert not np.allclose(nr[..., :rot], n0[..., :rot])


def pin_qk_partner_weight(L):
    D = 128
    rng = np.random.default_rng(4)
    x = np.zeros(D)
    x[D // 2:] = rng.normal(size=D // 2)
    xb = _to_bits(x)
    wb = _to_bits(np.concatenate([np.full(D // 2, 0.75), rng.uniform(1.0, 1.5, D // 2)]))
    wv = _bf16_value(wb)
    assert np.all(wv[:D // 2] != wv[D // 2:])
    cs = wl.host(wl.cos_sin_table(8, D, 1e4))
    p = 5
    inp = dict(qkv=np.ascontiguousarray(xb[None, :]), q_weight=wb, k_weight=wb, cos_sin=cs,
               positions=np.array([p], np.int64))
    _, ref, _ = _run_qk(L, inp, 1, 0, 0, D)
    xv = _bf16_value(xb)
    r = 1.0 / np.sqrt((xv * xv).sum() / D + float(np.float32(EPS)))
    c = cs[p, :D // 2].astype(np.float64)
    s = cs[p, D // 2:].astype(np.float64)
    partner = xv[D // 2:] * r * wv[D // 2:]    # n_{i+64} with w_{i+64}
    np.testing.assert_allclose(ref[0, 0, :D // 2], -partner * s, rtol=1e-13)
    np.testing.assert_allclose(ref[0, 0, D // 2:], partner * c, rtol=1e-13)


def pin_qk_pairing_index(L):
    D = 128
    x = np.zeros(D)
    x[3] = 1.0
    xb = _to_bits(x)
    wb = _to_bits(np.ones(D))
    cs = wl.host(wl.cos_sin_table(8, D, 1e4))
    inp = dict(qkv=np.ascontiguousarray(xb[None, :]), q_weight=wb, k_weight=wb, cos_sin=cs,
               positions=np.array([3], np.int64))
    _, ref, _ = _run_qk(L, inp, 1, 0, 0, D, is_neox=True)
    assert set(np.nonzero(ref[0, 0])[0].tolist()) == {3, 67}
    _, ref, _ = _run_qk(L, inp, 1, 0, 0, D, is_neox=False)
    assert set(np.nonzero(ref[0, 0])[0].tolist()) == {2, 3}
    n3 = ref[0, 0, 3] / cs[3, 1]          # the lone normalised input
    np.testing.assert_allclose(ref[0, 0, 2], -n3 * cs[3, D // 2 + 1], rtol=1e-13)


def pin_qk_v_untouched(L):
    T, Hq, Hk, Hv, D = 5, 2, 1, 3, 128
    inp = _qk_inputs(T, Hq, Hk, Hv, D)
    out, _, _ = _run_qk(L, inp, Hq, Hk, Hv, D)
    a = out.reshape(T, -1, D)[:, Hq + Hk:]
    b = inp["qkv"].reshape(T, -1, D)[:, Hq + Hk:]
    assert np.array_equal(a, b)
    inplace = inp["qkv"].copy()
    oracle.qk_norm_rope(inplace, Hq, Hk, Hv, D, EPS, inp["q_weight"], inp["k_weight"],
                        inp["cos_sin"], inp["positions"], out=inplace, _lib=L)
    assert np.array_equal(inplace, out)


# ---------------------------------------------------------------------------
# DSV4 operator
# ---------------------------------------------------------------------------

def _hand_entry():
    """584-byte entry for kv = 1 everywhere, pos 0, block weights below.

    r = 1/sqrt(1 + eps) = 0.9999995; n_j = r w_j.  Per block (w, e, scaled):
      w=1   e=-8  (1.75 >= n > 0.875)   n*2^8  = 255.99987 -> 256 = 0x78
      w=2   e=-7                          n*2^7  = 255.99987 -> 0x78
      w=4   e=-6                          n*2^6  -> 0x78
      w=8   e=-5                          n*2^5  -> 0x78
      w=0.5 e=-9                          n*2^9  -> 0x78
      w=3   e=-7  (3.5 >= 2.9999985)      n*2^7  = 383.9998 -> 384 = 0x7c
      w=5   e=-6  (7 >= 4.9999975 > 3.5)  n*2^6  = 319.9998 -> 320 = 0x7a
    RoPE dims (w = 1, pos 0 is the identity): bf16(0.9999995) = 1.0 = 0x3f80.
    """
    codes = [0x78] * (5 * 64) + [0x7C] * 64 + [0x7A] * 64
    rope = [0x80, 0x3F] * 64
    exps = [119, 120, 121, 122, 118, 120, 121]
    return np.array(codes + rope + exps + [0], np.uint8)


def pin_dsv4_hand_entry(L):
    block_w = [1.0, 2.0, 4.0, 8.0, 0.5, 3.0, 5.0, 1.0]
    kvw = _to_bits(np.repeat(block_w, 64))
    ones = _to_bits(np.ones(512))
    cs = wl.host(wl.cos_sin_table(4, 64, 1e4))
    cache = np.full((3, 4, 584), wl.SENTINEL, np.uint8)
    # token 0 has no slot (-1): it must leave the cache alone
    res = oracle.dsv4(np.ascontiguousarray(np.tile(ones, 2).reshape(2, 1, 512)),
                      np.ascontiguousarray(np.tile(ones, 2).reshape(2, 512)), EPS, ones, kvw,
                      cs, np.array([0, 0], np.int64), np.array([-1, 5], np.int64), cache,
                      _lib=L)
    flat = cache.reshape(-1)
    entry = flat[5 * 584:6 * 584]
    assert np.array_equal(entry, _hand_entry()), np.nonzero(entry != _hand_entry())[0][:8]
    rest = np.concatenate([flat[:5 * 584], flat[6 * 584:]])
    assert np.all(rest == wl.SENTINEL)
    assert np.all(res["q"] == 0x3F80)


def pin_dsv4_skip_and_addressing(L):
    inp = _dsv4_inputs(6, 2, num_blocks=4, block_size=4)
    inp["slot_mapping"] = np.array([3, -1, 15, 0, -1, 9], np.int64)
    a = _run_dsv4(L, inp, want_ref=False)
    flat = a["cache"].reshape(-1)
    written = np.zeros(flat.size, bool)
    for s in (3, 15, 0, 9):
        written[s * 584:(s + 1) * 584] = True
    assert np.all(flat[~written] == wl.SENTINEL)
    assert flat[3 * 584 + 583] == 0 and flat[15 * 584 + 583] == 0
    # q rows of skipped tokens are still processed
    assert not np.array_equal(a["q"][1], inp["q"][1])
    # the same slots addressed through another block size land on the same bytes
    inp2 = dict(inp, kv_cache=np.full((2, 8, 584), wl.SENTINEL, np.uint8))
    b = _run_dsv4(L, inp2, want_ref=False)
    assert np.array_equal(b["cache"].reshape(-1), flat)


def pin_dsv4_q_textbook(L):
    T, H = 3, 2
    inp = _dsv4_inputs(T, H)
    r0 = _run_dsv4(L, dict(inp, positions=np.zeros(T, np.int64)))
    want0 = _textbook(inp["q"].reshape(-1, 512), inp["q_weight"], 512).reshape(T, H, 512)
    np.testing.assert_allclose(r0["q_ref"], want0, rtol=1e-12)
    r = _run_dsv4(L, inp)
    cs = inp["cos_sin"][inp["positions"]][:, None, :]
    want = _complex_rotate(r0["q_ref"], cs, False, 448, 64)
    assert np.all(np.abs(r["q_ref"] - want) <= 1e-14 * r["q_mag"] + 1e-300)
    assert np.array_equal(r["q_ref"][..., :448], r0["q_ref"][..., :448])
    assert _is_nearest_bf16(r["q"], r["q_ref"]).all()
    kv0 = _textbook(inp["kv"], inp["kv_weight"], 512)
    np.testing.assert_allclose(r0["kv_ref"], kv0, rtol=1e-12)
    np.testing.assert_allclose(r["kv_ref"], _complex_rotate(kv0, cs[:, 0], False, 448, 64),
                               rtol=1e-12, atol=1e-15)


def pin_dsv4_kv_decisions(L):
    """Exponents and codes are decided on the unrounded normalised values
    (reading R5): the exponent is the smallest e with 448 * 2^e >= the block's
    exact amax, and each code is the e4m3 value nearest to the exact n * 2^-e,
    both found by exhaustive search in rational arithmetic."""
    T = 12
    inp = _dsv4_inputs(T, 1, num_blocks=4, block_size=4)
    r = _run_dsv4(L, inp)
    ent = r["cache"].reshape(-1, 584)[inp["slot_mapping"]]
    n64 = r["kv_ref"][:, :448].reshape(T, 7, 64)
    amax = np.abs(n64).max(-1)
    for t in range(T):
        for b in range(7):
            e = brute_ue8m0_exponent(float(amax[t, b]))
            byte = min(max(e + 127, 0), 254)
            assert ent[t, 576 + b] == byte
            want = [brute_e4m3_code(math.ldexp(float(v), -(byte - 127))) for v in n64[t, b]]
            assert np.array_equal(ent[t, 64 * b:64 * (b + 1)], np.array(want, np.uint8)), (t, b)
    rope = np.ascontiguousarray(ent[:, 448:576]).view(np.uint16)
    assert _is_nearest_bf16(rope, r["kv_ref"][:, 448:]).all()
    assert np.all(ent[:, 583] == 0)


def pin_dsv4_decisions_single_rounding(L):
    """Codes are rounded once, from the exact n * 2^-e (reading R5), not from
    an fp32 copy of it.  kv = 1 everywhere and eps = 2^-30 make r = (1 +
    2^-30)^-1/2, a hair below 1.  Block 0 has weights 1.75 (so e = -8) and
    19 * 2^-12, whose scaled value 1.1875 r lies 2^-31 (relative) below the
    midpoint of codes 0x39 (1.125) and 0x3a (1.25): rounding once gives 0x39;
    rounding to fp32 first lands on the midpoint and ties to the even 0x3a."""
    w = np.ones(512)
    w[0] = 1.75
    w[1] = 19 * 2.0**-12
    ones = _to_bits(np.ones(512))
    cache = np.full((1, 1, 584), wl.SENTINEL, np.uint8)
    res = oracle.dsv4(np.ascontiguousarray(ones.reshape(1, 1, 512)),
                      np.ascontiguousarray(ones.reshape(1, 512)), 2.0**-30, ones, _to_bits(w),
                      wl.host(wl.cos_sin_table(1, 64, 1e4)), np.zeros(1, np.int64),
                      np.zeros(1, np.int64), cache, want_ref=True, _lib=L)
    ent = cache.reshape(-1)
    v = math.ldexp(float(res["kv_ref"][0, 1]), 8)
    assert brute_e4m3_code(v) == 0x39 and brute_e4m3_code(float(np.float32(v))) == 0x3A
    assert ent[576] == 119 and ent[0] == 0x7E
    assert ent[1] == 0x39
    # The exponent too is decided on the exact amax: with x_0 = 1 - 2^-8 and
    # eps = 511 * 2^-25 - 2^-40 (both exact in bf16 / fp32), mean(x^2) + eps =
    # 1 - 2^-40, so r exceeds 1 by about 2^-41 and block 1's amax 1.75 r lies
    # just above 448 * 2^-8: e = -7 (byte 120).  Its fp32 copy is 1.75 (e = -8).
    x = np.ones(512)
    x[0] = 1 - 2.0**-8
    w = np.ones(512)
    w[64] = 1.75
    eps = 511 * 2.0**-25 - 2.0**-40
    assert float(np.float32(eps)) == eps
    cache = np.full((1, 1, 584), wl.SENTINEL, np.uint8)
    res = oracle.dsv4(np.ascontiguousarray(ones.reshape(1, 1, 512)),
                      np.ascontiguousarray(_to_bits(x).reshape(1, 512)), eps, ones, _to_bits(w),
                      wl.host(wl.cos_sin_table(1, 64, 1e4)), np.zeros(1, np.int64),
                      np.zeros(1, np.int64), cache, want_ref=True, _lib=L)
    amax = float(np.abs(res["kv_ref"][0, 64:128]).max())
    assert amax > 1.75 and float(np.float32(amax)) == 1.75
    assert brute_ue8m0_exponent(amax) == -7
    assert cache.reshape(-1)[577] == 120


def pin_dsv4_exp_margin(L):
    """The exponent margin the comparison relies on: for every block, the
    relative distance of the exact amax to the nearer boundary 448 * 2^k that
    brackets its exponent, in rational arithmetic; hand values at and near
    boundaries; an all-zero block has no boundary."""
    T = 10
    inp = _dsv4_inputs(T, 1, num_blocks=4, block_size=4)
    inp["kv"][3, :64] = 0                      # token 3, block 0: all zero
    r = _run_dsv4(L, inp)
    amax = np.abs(r["kv_ref"][:, :448].reshape(T, 7, 64)).max(-1)
    want = np.array([[brute_exponent_margin(float(a)) for a in row] for row in amax])
    got = r["exp_margin"]
    assert np.isinf(got[3, 0]) and np.isinf(want[3, 0])
    fin = np.isfinite(want)
    assert np.array_equal(np.isfinite(got), fin)
    np.testing.assert_allclose(got[fin], want[fin], rtol=1e-12, atol=0)
    assert L.orc_exponent_margin(448.0) == 0.0
    assert L.orc_exponent_margin(3.5) == 0.0
    m = L.orc_exponent_margin(3.5 * (1 + 2.0**-10))     # just above 448 * 2^-7
    assert abs(m - 2.0**-10 / (1 + 2.0**-10)) <= 1e-15
    m = L.orc_exponent_margin(448.0 * 0.75)             # midway (in ratio) of [224, 448]
    assert abs(m - 1.0 / 3.0) <= 1e-15
    assert math.isinf(L.orc_exponent_margin(0.0))


def _term_magnitudes(n0, cs_rows, neox, off, rot):
    """Sum of the magnitudes of the terms forming each rotated output, from
    the unrotated values n0: with za = |x| + i|y| (the pair) and wa = |c| +
    i|s| (the table row), the first element's terms sum to Re(za conj(wa)) and
    the second's to Im(za wa); dims outside the rotation keep |n0|."""
    half = rot // 2
    c = np.abs(cs_rows[..., :half].astype(np.float64))
    s = np.abs(cs_rows[..., half:rot].astype(np.float64))
    part = np.abs(n0[..., off:off + rot])
    za = (part[..., :half] + 1j * part[..., half:]) if neox else \
        (part[..., 0::2] + 1j * part[..., 1::2])
    wa = c + 1j * s
    first, second = (za * np.conj(wa)).real, (za * wa).imag
    out = np.abs(n0).copy()
    if neox:
        out[..., off:off + half], out[..., off + half:off + rot] = first, second
    else:
        out[..., off:off + rot:2], out[..., off + 1:off + rot:2] = first, second
    return out


def pin_qk_mag(L):
    """The magnitude sums the comparison's cancellation term uses, for full
    and partial rotation, both pairings, against the textbook RMSNorm
    (torch) and a complex-number form of the rotation's terms."""
    T, Hq, Hk, Hv = 3, 2, 1, 1
    pos = np.array([0, 9, 3000], np.int64)
    for D, rot, neox in ((128, 128, True), (64, 32, False), (256, 64, True)):
        d = wl.make_qk(T, Hq, Hk, Hv, D, 1e4, 4096, "uniform", 50 + D + rot, rotary_dim=rot)
        qkv, qw, kw = wl.bf16_bits(d["qkv"]), wl.bf16_bits(d["q_weight"]), wl.bf16_bits(d["k_weight"])
        cs = wl.host(d["cos_sin"])
        _, ref, mag = oracle.qk_norm_rope(qkv, Hq, Hk, Hv, D, EPS, qw, kw, cs, pos, is_neox=neox,
                                          rot_dim=rot, want_ref=True, nthreads=1, _lib=L)
        x = qkv.reshape(T, Hq + Hk + Hv, D)
        n0 = np.concatenate([
            _textbook(x[:, :Hq].copy(), qw, D, EPS).reshape(T, Hq, D),
            _textbook(x[:, Hq:Hq + Hk].copy(), kw, D, EPS).reshape(T, Hk, D)], axis=1)
        want = _term_magnitudes(n0, cs[pos][:, None, :], neox, 0, rot)
        np.testing.assert_allclose(mag, want, rtol=1e-12, atol=1e-300)
        assert np.all(np.abs(ref) <= mag * (1 + 1e-12))
        np.testing.assert_allclose(mag[0], np.abs(n0[0]), rtol=1e-12)   # position 0


def pin_dsv4_mag(L):
    """The same magnitude sums for the DSV4 q rows and kv vector (interleaved
    rotation of dims 448..511)."""
    T, H = 4, 2
    inp = _dsv4_inputs(T, H)
    r = _run_dsv4(L, inp)
    cs = inp["cos_sin"][inp["positions"]]
    n0q = _textbook(inp["q"].reshape(-1, 512), inp["q_weight"], 512).reshape(T, H, 512)
    np.testing.assert_allclose(r["q_mag"], _term_magnitudes(n0q, cs[:, None, :], False, 448, 64),
                               rtol=1e-12, atol=1e-300)
    n0k = _textbook(inp["kv"], inp["kv_weight"], 512)
    np.testing.assert_allclose(r["kv_mag"], _term_magnitudes(n0k, cs, False, 448, 64),
                               rtol=1e-12, atol=1e-300)


def pin_slicing_and_threads(L):
    inp = _dsv4_inputs(10, 3, num_blocks=8, block_size=4)
    full = _run_dsv4(L, inp, nthreads=1, want_ref=False)
    thr = _run_dsv4(L, inp, nthreads=4, want_ref=False)
    assert np.array_equal(full["q"], thr["q"]) and np.array_equal(full["cache"], thr["cache"])
    cache = inp["kv_cache"].copy()
    qs = []
    for a, b in ((0, 4), (4, 10)):
        part = {k: (v[a:b].copy() if k in ("q", "kv", "positions", "slot_mapping") else v)
                for k, v in inp.items()}
        part["kv_cache"] = cache
        res = oracle.dsv4(part["q"], part["kv"], EPS, part["q_weight"], part["kv_weight"],
                          part["cos_sin"], part["positions"], part["slot_mapping"], cache,
                          nthreads=2, _lib=L)
        qs.append(res["q"])
    assert np.array_equal(np.concatenate(qs), full["q"]) and np.array_equal(cache, full["cache"])


def pin_gather_hand_entry(L):
    """The hand-derived entry reads back as the block weights exactly:
    0x78 = 256, 0x7c = 384, 0x7a = 320 times 2^(byte - 127)."""
    cache = np.full((3, 4, 584), wl.SENTINEL, np.uint8)
    cache.reshape(-1)[5 * 584:6 * 584] = _hand_entry()
    out = oracle.dsv4_gather(cache, np.array([5, -1], np.int64), _lib=L)
    want = np.repeat([1.0, 2.0, 4.0, 8.0, 0.5, 3.0, 5.0, 1.0], 64)
    assert np.array_equal(_bf16_value(out[0]), want)
    assert np.all(out[1] == 0)


def pin_gather_round_trip(L):
    """Insert then read back: each dequantised value is within half an e4m3
    step of the exact value the codes were taken from (2^-4 relative for
    normal codes, 2^(e-10) absolute below), and the rotary dims come back as
    the nearest bf16 of the exact values."""
    T = 16
    inp = _dsv4_inputs(T, 1, num_blocks=8, block_size=4)
    r = _run_dsv4(L, inp)
    out = oracle.dsv4_gather(r["cache"], inp["slot_mapping"], _lib=L)
    got = _bf16_value(out)
    ent = r["cache"].reshape(-1, 584)[inp["slot_mapping"]]
    e = ent[:, 576:583].astype(np.int64) - 127
    f32 = r["kv_ref"][:, :448].reshape(T, 7, 64)
    scale = np.ldexp(1.0, e)[:, :, None]
    err = np.abs(got[:, :448].reshape(T, 7, 64) - f32)
    bound = np.maximum(np.abs(f32) * 2.0 ** -4, scale * 2.0 ** -10)
    assert np.all(err <= bound * (1 + 1e-12))
    assert _is_nearest_bf16(out[:, 448:], r["kv_ref"][:, 448:]).all()


ALL_PINS = [
    pin_bf16_value_and_roundtrip, pin_bf16_vs_torch, pin_bf16_single_rounding,
    pin_e4m3_decode_vs_torch, pin_e4m3_roundtrip, pin_e4m3_vs_torch,
    pin_ue8m0_hand, pin_ue8m0_bruteforce,
    pin_qk_textbook_rmsnorm, pin_qk_all_equal_row, pin_qk_rope_complex, pin_qk_rope_partial,
    pin_qk_partner_weight, pin_qk_pairing_index, pin_qk_v_untouched,
    pin_dsv4_hand_entry, pin_dsv4_skip_and_addressing, pin_dsv4_q_textbook,
    pin_dsv4_kv_decisions, pin_dsv4_decisions_single_rounding, pin_dsv4_exp_margin, pin_qk_mag,
    pin_dsv4_mag,
    pin_slicing_and_threads, pin_gather_hand_entry, pin_gather_round_trip,
]
