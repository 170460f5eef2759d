"""CPU model of the cache write's rounding decision, checked with exact
rational arithmetic.

The write kernels compute a rotated (bf16 cache) or scaled (FP8 cache) value
first in fp32, y, together with a bound e on its distance from the exact
value, and keep the rounding of y when y - e and y + e round to the same
code; otherwise they recompute from fp64 products.  This test replays that
decision step by step in fp32 (numpy float32 and exactly rounded fused
multiply-adds) and asserts that whenever the decision is taken in fp32, the
code equals the correctly rounded code of the exact value -- for bf16
rotations (random pairs and pairs built to cancel) and for E4M3 codes of V
(scaled) and K (rotated, then scaled).  No GPU: it checks the argument the
kernels rely on, not the kernels (their outputs are compared with the oracle
in tests/test_gpu_write.py and tests/test_gpu_fp8.py)."""
import bisect
import math
from fractions import Fraction as Q

import numpy as np

F32 = np.float32


def f32_round(q: Q) -> np.float32:
    """Nearest float32 to the rational q, ties to even."""
    f = F32(float(q))
    best = None
    for c in (f, np.nextafter(f, F32(np.inf)), np.nextafter(f, F32(-np.inf))):
        key = (abs(Q(float(c)) - q), int(np.array(c, F32).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def fma32(a, b, c) -> np.float32:
    return f32_round(Q(float(a)) * Q(float(b)) + Q(float(c)))


def bf16_bits_of_f32(x: np.float32) -> int:
    """Round-to-nearest-even bf16 bits of a finite float32."""
    b = int(np.array(x, F32).view(np.uint32))
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) & 0xFFFF


def bf16_value(bits: int) -> float:
    return float(np.array(bits << 16, np.uint32).view(F32))


def bf16_bits_exact(q: Q) -> int:
    """Nearest bf16 to the rational q, ties to even."""
    c0 = bf16_bits_of_f32(F32(float(q)))
    best = None
    for c in ((c0 - 1) & 0xFFFF, c0, (c0 + 1) & 0xFFFF):
        v = bf16_value(c)
        if not math.isfinite(v):
            continue
        key = (abs(Q(v) - q), c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def _e4m3_table():
    vals = []
    for code in range(256):
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            continue  # NaN
        v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        vals.append((-v if s else v, code))
    vals.sort()
    return [v for v, _ in vals], [c for _, c in vals]


E4_VALS, E4_CODES = _e4m3_table()


def e4m3_exact(q: Q) -> float:
    """Nearest E4M3 value to the rational q, ties to the even code, saturating
    at +-448 (the value, so +0 and -0 compare equal)."""
    if q >= 448:
        return 448.0
    if q <= -448:
        return -448.0
    i = bisect.bisect_left(E4_VALS, float(q))
    best = None
    for j in (i - 1, i, i + 1):
        if 0 <= j < len(E4_VALS):
            key = (abs(Q(E4_VALS[j]) - q), E4_CODES[j] & 1)
            if best is None or key < best[0]:
                best = (key, E4_VALS[j])
    return best[1]


def e4m3_of_f32(x: np.float32) -> float:
    return e4m3_exact(Q(float(x)))


def bf16_input(rng, scale=1.0) -> np.float32:
    return F32(bf16_value(bf16_bits_of_f32(F32(rng.normal() * scale))))


def rotation_case(rng, cancel):
    """(u, w, c64, t64): rotated element u*c + w*t; `cancel` builds u = the
    bf16 nearest tan(angle) against w = -1, so u*cos - sin nearly cancels."""
    ang = rng.uniform(0.0, 60000.0)
    c64, s64 = math.cos(ang), math.sin(ang)
    if cancel:
        u = F32(bf16_value(bf16_bits_of_f32(F32(math.tan(ang)))))
        return u, F32(-1.0), c64, s64
    t64 = -s64 if rng.random() < 0.5 else s64
    return bf16_input(rng), bf16_input(rng), c64, t64


def test_bf16_rotation_decision_agrees_with_exact_rounding():
    rng = np.random.default_rng(1)
    taken = fallback_random = 0
    for n in range(1500):
        cancel = n % 2 == 1
        u, w, c64, t64 = rotation_case(rng, cancel)
        c32, t32 = F32(c64), F32(t64)
        y = fma32(u, c32, F32(w * t32))
        e = fma32(F32(F32(abs(y) + abs(u)) + abs(w)), F32(2.0 ** -22), F32(2.0 ** -126))
        lo, hi = bf16_bits_of_f32(F32(y - e)), bf16_bits_of_f32(F32(y + e))
        exact = bf16_bits_exact(Q(float(u)) * Q(c64) + Q(float(w)) * Q(t64))
        if lo == hi:
            taken += 1
            assert lo == exact, (u, w, c64, t64)
        elif not cancel:
            fallback_random += 1
    assert taken > 1000                 # the fp32 decision is the common path
    assert fallback_random <= 15        # and the fp64 one rare on random pairs (~1 %)


def midpoint_scale(x: float, rng) -> np.float32:
    """A positive fp32 scale sc with x / sc within ~2^-24 of a midpoint of two
    adjacent E4M3 values (a rounding boundary), or 0 if none is usable."""
    k = int(rng.integers(len(E4_VALS) // 2, len(E4_VALS) - 1))  # positive values
    mid = (E4_VALS[k] + E4_VALS[k + 1]) / 2
    if x == 0.0 or mid <= 0.0:
        return F32(0.0)
    sc = F32(abs(x) / mid)
    return sc if 1e-30 < float(sc) < 1e30 else F32(0.0)


def test_e4m3_v_decision_agrees_with_exact_rounding():
    rng = np.random.default_rng(2)
    taken = boundary_cases = 0
    for n in range(1000):
        x = bf16_input(rng, 2.0)
        sc = midpoint_scale(float(x), rng) if n % 2 else F32(0.0)
        if float(sc) == 0.0:
            sc = F32(rng.uniform(0.5, 1.5) * 4 / 448)
        else:
            boundary_cases += 1
        is32 = F32(1.0) / sc
        y = F32(x * is32)
        e = fma32(F32(F32(abs(x) * abs(is32)) + abs(y)), F32(2.0 ** -22), F32(2.0 ** -126))
        lo, hi = e4m3_of_f32(F32(y - e)), e4m3_of_f32(F32(y + e))
        if lo == hi:
            taken += 1
            assert lo == e4m3_exact(Q(float(x)) / Q(float(sc))), (x, sc)
    assert boundary_cases > 400 and taken > 400


def test_e4m3_exact_ties_always_take_the_fp64_quotient():
    """x / sc exactly on an E4M3 midpoint (sc an odd 19-bit integer times a
    power of two): the fp32 product cannot tell which side of the tie it is
    on, so the margin must always straddle the midpoint and hand the code to
    the fp64 quotient, whose single rounding lands on the tie exactly."""
    rng = np.random.default_rng(4)
    mids = [(a + b) / 2 for a, b in zip(E4_VALS, E4_VALS[1:]) if b > 0 and a >= 0]
    n = 0
    while n < 500:
        mid = mids[int(rng.integers(0, len(mids)))]
        sc = float(int(rng.integers(2 ** 18, 2 ** 19)) | 1) * 2.0 ** int(rng.integers(-30, -20))
        x = mid * sc
        if F32(x) != x or F32(sc) != sc:
            continue
        n += 1
        x, sc = F32(x), F32(sc)
        is32 = F32(1.0) / sc
        y = F32(x * is32)
        e = fma32(F32(F32(abs(x) * abs(is32)) + abs(y)), F32(2.0 ** -22), F32(2.0 ** -126))
        assert e4m3_of_f32(F32(y - e)) != e4m3_of_f32(F32(y + e)), (x, sc)
        assert float(x) / float(sc) == mid  # the fp64 quotient is the tie itself


def test_e4m3_k_decision_agrees_with_exact_rounding():
    rng = np.random.default_rng(3)
    taken = 0
    for n in range(1000):
        u, w, c64, t64 = rotation_case(rng, n % 4 == 1)
        sc = midpoint_scale(float(u) * c64 + float(w) * t64, rng) if n % 2 == 0 else F32(0.0)
        if float(sc) == 0.0:
            sc = F32(rng.uniform(0.5, 1.5) * 4 / 448)
        is32 = F32(1.0) / sc
        c32, t32 = F32(c64), F32(t64)
        rr = fma32(u, c32, F32(w * t32))
        y = F32(rr * is32)
        inner = F32(F32(abs(u) + abs(w)) + F32(2.0 * abs(rr)))
        e = fma32(F32(F32(abs(is32) * inner) + abs(y)), F32(2.0 ** -22), F32(2.0 ** -126))
        lo, hi = e4m3_of_f32(F32(y - e)), e4m3_of_f32(F32(y + e))
        if lo == hi:
            taken += 1
            exact = (Q(float(u)) * Q(c64) + Q(float(w)) * Q(t64)) / Q(float(sc))
            assert lo == e4m3_exact(exact), (u, w, c64, t64, sc)
    assert taken > 400
