"""Comparison of the CUDA path's outputs with the oracle's (test-side only).

Tolerances (derived in the design notes):
  * bf16 outputs: within one bf16 ulp of the oracle's unrounded fp64 result
    ``exact``.  The one allowance beyond that is for results that cancel:
    a value whose terms' magnitudes sum to ``mag`` (|n| for an unrotated
    element, |n_a c| + |n_b s| for a rotated one) may differ from ``exact`` by
    up to ulp + 2^-15 mag, but only where it cancels by at least
    CANCEL_BITS bits (|exact| < 2^-CANCEL_BITS mag).  2^-15 bounds the
    relative fp32 error of the terms (a 512-term sum of squares, a reciprocal
    square root, two products and a fused multiply-add: below (D + 8) 2^-24);
    such an error can reach a full ulp of the result only where the result is
    that much smaller than its terms.  Every value that needs the allowance is
    counted (``beyond_ulp``) and reported with the shallowest cancellation
    among them.
  * UE8M0 exponent bytes, slot placement, untouched bytes, pad: bit-exact;
    the only excused exponent mismatches are blocks whose exact amax lies
    within 2^-20 (relative) of a power-of-two boundary, and they are counted
    (the tests assert none occur at their seeds).
  * e4m3 codes: >= 99.99 % bit-exact, the rest at most one code apart
    (codes compared in value order, +0 and -0 equal).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

EXP_TIE_MARGIN = 2.0 ** -20
CODE_EXACT_MIN = 0.9999
MAG_TERM = 2.0 ** -15
CANCEL_BITS = 6


def bf16_values(bits: np.ndarray) -> np.ndarray:
    with np.errstate(invalid="ignore"):
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (2^-133 below the normal range)."""
    _, e = np.frexp(np.abs(x))          # |x| in [2^(e-1), 2^e)
    return np.where(x == 0, 2.0 ** -133, np.ldexp(1.0, np.maximum(e - 8, -133)))


@dataclass
class Bf16Report:
    n: int = 0
    exact: int = 0
    bad: int = 0
    beyond_ulp: int = 0            # within tolerance only through the cancellation allowance
    min_cancel_bits: float = math.inf  # shallowest cancellation among those (log2 mag/|exact|)
    max_ulps: float = 0.0          # largest |gpu - exact| in ulps of exact
    first_bad: list = field(default_factory=list)

    def add(self, gpu_bits, oracle_bits, ref, mag):
        g = gpu_bits.ravel()
        o = oracle_bits.ravel()
        self.n += g.size
        diff = np.nonzero(g != o)[0]
        self.exact += g.size - diff.size
        if diff.size == 0:
            return
        r = ref.ravel()[diff]
        m = mag.ravel()[diff]
        err = np.abs(bf16_values(g[diff]) - r)
        ulp = ulp_bf16(r)
        within = err <= ulp
        cancels = np.abs(r) < 2.0 ** -CANCEL_BITS * m
        excused = ~within & cancels & (err <= ulp + MAG_TERM * m)
        badm = ~(within | excused)
        self.max_ulps = max(self.max_ulps, float(np.max(err / ulp)))
        if excused.any():
            self.beyond_ulp += int(excused.sum())
            with np.errstate(divide="ignore"):
                depth = np.log2(m[excused] / np.abs(r[excused]))
            self.min_cancel_bits = min(self.min_cancel_bits, float(np.min(depth)))
        if badm.any():
            self.bad += int(badm.sum())
            for i in np.nonzero(badm)[0][:5]:
                self.first_bad.append((int(diff[i]), float(bf16_values(g[diff[i]:diff[i] + 1])[0]),
                                       float(r[i]), float(m[i])))

    def check(self, what=""):
        assert self.bad == 0, f"{what}: {self.bad} bf16 values outside tolerance, e.g. {self.first_bad}"

    @property
    def exact_frac(self):
        return self.exact / max(self.n, 1)

    def summary(self) -> str:
        s = (f"{self.n} bf16 values: {self.exact_frac:.6f} equal to the oracle's rounding, "
             f"max {self.max_ulps:.3f} ulp, {self.beyond_ulp} beyond 1 ulp")
        if self.beyond_ulp:
            s += f" (each a cancellation of >= {self.min_cancel_bits:.1f} bits)"
        return s


def code_order(c: np.ndarray) -> np.ndarray:
    c = c.astype(np.int32)
    return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)


@dataclass
class CacheReport:
    entries: int = 0
    codes: int = 0
    codes_exact: int = 0
    codes_far: int = 0
    exp_mismatch_ties: int = 0
    exp_mismatch_bad: int = 0
    rope: Bf16Report = field(default_factory=Bf16Report)

    def summary(self) -> str:
        frac = self.codes_exact / self.codes if self.codes else 1.0
        return (f"{self.entries} entries: e4m3 codes {frac:.7f} exact "
                f"({self.codes - self.codes_exact} one code apart), exponent near-ties "
                f"{self.exp_mismatch_ties}; rotary part: {self.rope.summary()}")

    def check(self, what=""):
        assert self.exp_mismatch_bad == 0, f"{what}: {self.exp_mismatch_bad} exponent bytes differ"
        assert self.codes_far == 0, f"{what}: {self.codes_far} e4m3 codes more than one code apart"
        if self.codes:
            frac = self.codes_exact / self.codes
            assert frac >= CODE_EXACT_MIN, f"{what}: only {frac:.6f} of e4m3 codes bit-exact"
        self.rope.check(what + " (rotary bf16 in cache)")


def compare_cache(gpu_cache: np.ndarray, ora_cache: np.ndarray, slots: np.ndarray,
                  kv_ref: np.ndarray, kv_mag: np.ndarray, margin: np.ndarray,
                  rep: CacheReport | None = None, check_untouched=True) -> CacheReport:
    """Compare two caches: mapped entries with tolerances, the rest bit-exact.

    slots, kv_ref, kv_mag, margin are per token (slot -1 = no entry)."""
    rep = rep or CacheReport()
    g = gpu_cache.reshape(-1, 584)
    o = ora_cache.reshape(-1, 584)
    mapped = slots >= 0
    s = slots[mapped]
    if check_untouched:
        untouched = np.ones(g.shape[0], bool)
        untouched[s] = False
        assert np.array_equal(g[untouched], o[untouched]), "bytes outside mapped entries changed"
    ge, oe = g[s], o[s]
    rep.entries += s.size
    # exponent bytes and pad: exact, apart from near-tie blocks
    assert np.array_equal(ge[:, 583], oe[:, 583]), "pad byte"
    gexp, oexp = ge[:, 576:583], oe[:, 576:583]
    mism = gexp != oexp
    tie = margin[mapped] < EXP_TIE_MARGIN
    rep.exp_mismatch_ties += int((mism & tie).sum())
    rep.exp_mismatch_bad += int((mism & ~tie).sum())
    # codes, excluding blocks whose exponent legitimately differs
    gc = ge[:, :448].reshape(-1, 7, 64)
    oc = oe[:, :448].reshape(-1, 7, 64)
    keep = ~mism
    gck, ock = gc[keep], oc[keep]
    rep.codes += gck.size
    rep.codes_exact += int((gck == ock).sum())
    rep.codes_far += int((np.abs(code_order(gck) - code_order(ock)) > 1).sum())
    # rotary bf16
    grope = np.ascontiguousarray(ge[:, 448:576]).view(np.uint16)
    orope = np.ascontiguousarray(oe[:, 448:576]).view(np.uint16)
    rep.rope.add(grope, orope, kv_ref[mapped][:, 448:], kv_mag[mapped][:, 448:])
    return rep
