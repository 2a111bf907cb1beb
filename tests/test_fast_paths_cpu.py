"""Host models of the kernels' float32 fast paths, checked against exact values.

The projection prologue and the SwiGLU epilogue take a BF16 rounding from a
float32 evaluation where that evaluation lies far from a BF16 midpoint, and
the prologue takes a row's absmax from the largest |x w|. These tests replay
those steps in numpy float32 on many seeded values and check each decision
against the rounding of the exactly computed value (Python floats and
fractions), so the error bounds the fast paths rely on are exercised on the
CPU as well as through the GPU parity tests.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

f32 = np.float32


def rn_bf16(v) -> float:
    """Round-to-nearest-even of a real (Fraction or float) to BF16 (8
    significant bits), for normal magnitudes."""
    v = Fraction(v)
    if v == 0:
        return 0.0
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = math.floor(math.log2(a))
    if Fraction(2) ** e > a:
        e -= 1
    if Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (e - 7)
    q = a / ulp
    n = math.floor(q)
    r = q - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return float(sign * n * ulp)


def bf16_of_f32(x: np.float32) -> float:
    """RN_bf16 of a float32 value."""
    return rn_bf16(Fraction(float(x)))


def far_from_midpoint(x: np.float32, units: int) -> bool:
    """The kernels' test: normal, finite, and the low 16 bits more than
    `units` float32 units away from 0x8000."""
    u = int(np.array([x], np.float32).view(np.uint32)[0])
    ex = u & 0x7F800000
    d = ((u & 0xFFFF) - (0x8000 - units)) & 0xFFFFFFFF
    return d >= 2 * units + 1 and ex != 0 and ex != 0x7F800000


def bf16_values(rng, n, scale):
    x = (rng.standard_normal(n) * scale).astype(np.float32)
    # keep the upper 16 bits: exact BF16 values
    return (x.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)


def near_midpoints(rng, n, units, lo_exp=-4, hi_exp=6):
    """Reals within `units` float32 units of BF16 midpoints (where the
    rounding decision is delicate)."""
    out = []
    for _ in range(n):
        e = int(rng.integers(lo_exp, hi_exp))
        mant = int(rng.integers(128, 256))                      # 8 significant bits
        mid = (mant + 0.5) * 2.0 ** (e - 7)                     # a BF16 midpoint
        off = float(rng.uniform(-units, units)) * 2.0 ** (e - 23)
        out.append((mid + off) * (1 if rng.random() < 0.5 else -1))
    return out


def test_swiglu_float_path_agrees_with_the_exact_value():
    # silu(g) u from float32 g, u: g u / (1 + e) for g >= 0, g u e / (1 + e)
    # for g < 0, e = exp(-|g|); the float evaluation decides where it is more
    # than 64 float32 units from a BF16 midpoint (and g > -80)
    rng = np.random.default_rng(11)
    g = np.concatenate([rng.standard_normal(6000) * 3, rng.standard_normal(2000) * 30,
                        rng.uniform(-79, 79, 2000)]).astype(np.float32)
    u = (rng.standard_normal(g.size) * 20).astype(np.float32)
    # and pairs whose value sits within a few float32 units of a BF16 midpoint
    g2 = (rng.standard_normal(4000) * 3).astype(np.float32)
    u2 = []
    for gi, target in zip(g2, near_midpoints(rng, g2.size, 120)):
        gd = float(gi)
        s_ = gd / (1.0 + math.exp(-gd)) if gd >= 0 else gd * math.exp(gd) / (1.0 + math.exp(gd))
        u2.append(target / s_ if s_ != 0 else 1.0)
    g = np.concatenate([g, g2])
    u = np.concatenate([u, np.array(u2, np.float32)])
    fast = slow = 0
    for gi, ui in zip(g, u):
        e = np.exp(f32(-abs(gi)), dtype=np.float32)
        r = f32(f32(gi * ui) / f32(f32(1) + e))
        if gi < 0:
            r = f32(r * e)
        if not (far_from_midpoint(r, 64) and gi > -80):
            slow += 1
            continue
        fast += 1
        gd, ud = float(gi), float(ui)
        # exact enough: double evaluation, 2^-50 relative, far inside the
        # 54-unit margin left by the fast-path test
        exact = gd * ud / (1.0 + math.exp(-gd)) if gd >= 0 else gd * ud * math.exp(gd) / (1.0 + math.exp(gd))
        assert bf16_of_f32(r) == rn_bf16(exact), (gi, ui, r, exact)
    # the targeted values land on both sides of the 64-unit margin
    assert fast > 11000 and slow > 1500, (fast, slow)


def test_norm_float_path_agrees_with_the_exact_value():
    # RN_bf16(xw * inv) for an exact float32 xw = x w and inv = hi + lo; the
    # float product p = RN(xw hi) decides where it is more than 4 units from
    # a BF16 midpoint
    rng = np.random.default_rng(12)
    x = bf16_values(rng, 20000, 2.0)
    w = (1 + 0.02 * rng.standard_normal(x.size)).astype(np.float32)
    w = (w.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    fast = 0
    for inv in (0.37123456789, 1.0 / math.sqrt(2.71828 + 1e-6), 3.1415926535):
        hi = f32(inv)
        lo = f32(inv - float(hi))
        inv_pair = Fraction(float(hi)) + Fraction(float(lo))
        # xw values whose product with inv sits near a BF16 midpoint
        near = [f32(t / inv) for t in near_midpoints(rng, 3000, 10, -3, 4)]
        near = [(f32(v), f32(1)) for v in near]
        for xi, wi in list(zip(x[:7000], w[:7000])) + near:
            xw = f32(xi * wi)
            assert Fraction(float(xw)) == Fraction(float(xi)) * Fraction(float(wi))  # exact
            p = f32(xw * hi)
            if not far_from_midpoint(p, 4) or xw == 0:
                continue
            fast += 1
            assert bf16_of_f32(p) == rn_bf16(Fraction(float(xw)) * inv_pair), (xi, wi, inv)
    assert fast > 20000


def test_row_absmax_from_the_largest_x_w():
    # the largest |RN_bf16(x_k w_k inv)| over a row is RN_bf16(max |x_k w_k| inv)
    rng = np.random.default_rng(13)
    for trial in range(40):
        x = bf16_values(rng, 512, 10 ** rng.uniform(-2, 2))
        w = (1 + 0.02 * rng.standard_normal(x.size)).astype(np.float32)
        w = (w.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
        inv = Fraction(float(f32(rng.uniform(0.05, 20.0))))
        xw = [Fraction(float(f32(a * b))) for a, b in zip(x, w)]
        by_element = max(abs(rn_bf16(v * inv)) for v in xw if v != 0)
        by_max = rn_bf16(max(abs(v) for v in xw) * inv)
        assert by_element == by_max, trial
