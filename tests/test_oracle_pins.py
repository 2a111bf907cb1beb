"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks one oracle function against a closed form, a hand-derived
fixture under tests/golden/, an invariant of the mathematics, or a brute force
by an independent library routine, so that a plausible slip (dropped term,
wrong sign or index, transposed operand, wrong rounding) fails at least one.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# independent helpers (not the oracle's code)
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(f):
    """Classic bit-level float32 -> bf16 round-to-nearest-even (finite inputs)."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = 0x7FFF + ((u >> 16) & 1)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f64(h):
    return (np.asarray(h, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_of(x):
    """bf16 bit pattern for exactly representable values."""
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


ALL_BF16 = np.arange(0, 0x7F80, dtype=np.uint32).astype(np.uint16)   # finite >= 0
ALL_BF16_VAL = bf16_bits_to_f64(ALL_BF16)


def bf16_nearest_bruteforce(x: float) -> int:
    """Exact RNE by search over every finite non-negative BF16 value."""
    sign = 0x8000 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    i = int(np.searchsorted(ALL_BF16_VAL, a))
    if i >= len(ALL_BF16_VAL):
        return sign | 0x7F80
    if ALL_BF16_VAL[i] == a:
        return sign | int(ALL_BF16[i])
    lo, hi = i - 1, i
    fa = Fraction(a)
    dlo = fa - Fraction(ALL_BF16_VAL[lo])
    if hi >= len(ALL_BF16_VAL):
        # above the largest finite value: compare with the halfway point to 2^128
        top = Fraction(2) ** 128
        return sign | (int(ALL_BF16[lo]) if fa - Fraction(ALL_BF16_VAL[lo]) < top - fa
                       or (fa - Fraction(ALL_BF16_VAL[lo]) == top - fa and ALL_BF16[lo] % 2 == 0)
                       else 0x7F80)
    dhi = Fraction(ALL_BF16_VAL[hi]) - fa
    if dlo < dhi:
        return sign | int(ALL_BF16[lo])
    if dhi < dlo:
        return sign | int(ALL_BF16[hi])
    return sign | int(ALL_BF16[lo] if ALL_BF16[lo] % 2 == 0 else ALL_BF16[hi])


# ---------------------------------------------------------------------------
# BF16 narrowing
# ---------------------------------------------------------------------------

def _golden_rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [p.strip() for p in line.split("|")]


def test_bf16_rne_golden():
    for expr, hexbits in _golden_rows("bf16_rne_cases.txt"):
        x = float(eval(expr))   # fixture values are plain arithmetic on literals
        got = int(oracle.bf16_from_f64(np.array([x]))[0])
        assert got == int(hexbits, 16), (expr, hex(got), hexbits)


def test_bf16_rne_matches_bitlevel_rule_on_floats():
    rng = np.random.default_rng(0)
    f = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 20000),
                        rng.standard_normal(2000).astype(np.float32)])
    f = f.astype(np.float32)
    # include exact ties: bf16 values plus half an ulp
    base = rng.standard_normal(2000).astype(np.float32)
    ties = ((base.view(np.uint32) & 0xFFFF0000) | 0x8000).view(np.float32)
    f = np.concatenate([f, ties])
    got = oracle.bf16_from_f64(f.astype(np.float64))
    assert np.array_equal(got, f32_to_bf16_bits(f))


def test_bf16_rne_matches_bruteforce_on_doubles():
    rng = np.random.default_rng(1)
    xs = rng.standard_normal(400) * 10.0 ** rng.integers(-40, 39, 400)
    got = oracle.bf16_from_f64(xs)
    for x, g in zip(xs, got):
        assert int(g) == bf16_nearest_bruteforce(float(x)), x


# ---------------------------------------------------------------------------
# Quantisation
# ---------------------------------------------------------------------------

def test_quant_golden_cases():
    for xs, sc, codes in _golden_rows("quant_cases.txt"):
        x = np.array([float(v) for v in xs.split()], dtype=np.float32)
        expect_q = np.array([int(v) for v in codes.split()], dtype=np.int8)
        if "/" in sc:
            a, b = sc.split("/")
            expect_s = np.float32(float(a)) / np.float32(float(b))
        else:
            expect_s = np.float32(float(sc))
        q, s = oracle.quant_rows(bf16_of(x)[None, :])
        assert s[0] == expect_s, (xs, s[0], expect_s)
        assert np.array_equal(q[0], expect_q), (xs, q[0], expect_q)


def test_quant_invariants_random_rows():
    rng = np.random.default_rng(2)
    for cols in (1, 7, 256, 5120):
        for scale in (1e-3, 1.0, 300.0):
            x = bf16_of(rng.standard_normal((4, cols)).astype(np.float32) * scale)
            q, s = oracle.quant_rows(x)
            xv = bf16_bits_to_f64(x)
            amax = np.abs(xv).max(axis=1)
            assert np.all(np.abs(q.astype(np.int32)) <= 127)
            assert np.all(q != -128)
            # the absmax element maps to +-127
            idx = np.abs(xv).argmax(axis=1)
            for r in range(4):
                assert abs(int(q[r, idx[r]])) == 127
                assert np.sign(q[r, idx[r]]) == np.sign(xv[r, idx[r]])
            # scale is absmax/127 up to float32 rounding
            np.testing.assert_allclose(s, amax / 127.0, rtol=1e-7)
            # reconstruction error at most half a step (plus float32 slack)
            err = np.abs(xv - q.astype(np.float64) * s[:, None].astype(np.float64))
            assert np.all(err <= s[:, None] * (0.5 + 1e-5))


def test_quant_rows_are_independent():
    rng = np.random.default_rng(3)
    x = bf16_of(rng.standard_normal((5, 300)).astype(np.float32) * np.array([[1], [10], [0.1], [3], [100]], dtype=np.float32))
    q, s = oracle.quant_rows(x)
    for r in range(5):
        qr, sr = oracle.quant_rows(x[r:r + 1])
        assert np.array_equal(qr[0], q[r]) and sr[0] == s[r]


# ---------------------------------------------------------------------------
# INT8 matmul and dequantisation
# ---------------------------------------------------------------------------

def test_matmul_i8_bruteforce():
    rng = np.random.default_rng(4)
    for (M, K, N) in ((1, 16, 3), (3, 256, 40), (16, 512, 7)):
        x = rng.integers(-127, 128, (M, K), dtype=np.int8)
        W = rng.integers(-127, 128, (N, K), dtype=np.int8)
        acc = oracle.matmul_i8(x, W)
        ref = x.astype(np.int64) @ W.astype(np.int64).T
        assert np.array_equal(acc, ref)
        # split additivity over K
        h = K // 2
        a0 = oracle.matmul_i8(x, W, 0, h)
        a1 = oracle.matmul_i8(x, W, h, K)
        assert np.array_equal(a0.astype(np.int64) + a1, ref)


def test_matmul_i8_extremes_fit_int32():
    K = 17408
    x = np.full((1, K), 127, dtype=np.int8)
    W = np.full((2, K), -127, dtype=np.int8)
    W[1] = 127
    acc = oracle.matmul_i8(x, W)
    assert acc[0, 0] == -127 * 127 * K and acc[0, 1] == 127 * 127 * K


def test_dequant_closed_forms():
    assert oracle.dequant(3, 0.5, 0.25) == np.float32(0.375)
    assert oracle.dequant(-7, 2.0, 0.125) == np.float32(-1.75)
    assert oracle.dequant(0, 3.3, 1e-3) == 0.0
    # the activation scale is applied first: float32(float32(a*sa)*sw)
    a, sa, sw = 123456789, np.float32(0.1), np.float32(0.3)
    first = np.float32(np.float32(np.float32(a) * sa) * sw)
    assert oracle.dequant(a, sa, sw) == first


def _exact(acc, sa, sw):
    return float(Fraction(int(acc)) * Fraction(float(sa)) * Fraction(float(sw)))


@pytest.mark.parametrize("k_splits", [1, 2, 4])
@pytest.mark.parametrize("with_res", [False, True])
def test_linear_within_error_bound_of_exact(k_splits, with_res):
    rng = np.random.default_rng(5 + k_splits)
    M, K, N = 3, 512, 33
    xq = rng.integers(-127, 128, (M, K), dtype=np.int8)
    xs = rng.uniform(0.001, 0.05, M).astype(np.float32)
    W = rng.integers(-127, 128, (N, K), dtype=np.int8)
    ws = rng.uniform(1e-3, 4e-3, N).astype(np.float32)
    res = bf16_of(rng.standard_normal((M, N)).astype(np.float32) * 4) if with_res else None
    y, acc = oracle.linear(xq, xs, W, ws, k_splits, res)
    ref_acc = xq.astype(np.int64) @ W.astype(np.int64).T
    assert np.array_equal(acc, ref_acc)
    yv = bf16_bits_to_f64(y)
    for m in range(M):
        for n in range(N):
            exact = _exact(ref_acc[m, n], xs[m], ws[n])
            if with_res:
                exact += float(bf16_bits_to_f64(res[m, n]))
            # bf16 half-ulp (at most 2^-8 relative) plus float32 slack of the few operations
            tol = abs(exact) * (2.0 ** -8 + 8 * 2.0 ** -24) + 1e-30 + (
                (abs(exact) + 50.0) * 8 * 2.0 ** -24 if k_splits > 1 or with_res else 0.0)
            assert abs(yv[m, n] - exact) <= tol, (m, n, yv[m, n], exact)


def test_linear_transposition_pinned():
    # W is [N, K]: output n must use row n of W. A single non-zero weight shows it.
    K, N = 32, 4
    W = np.zeros((N, K), dtype=np.int8)
    W[2, 5] = 10
    xq = np.zeros((1, K), dtype=np.int8)
    xq[0, 5] = 3
    y, acc = oracle.linear(xq, np.array([1.0], np.float32), W, np.ones(N, np.float32))
    assert acc.tolist() == [[0, 0, 30, 0]]
    assert bf16_bits_to_f64(y).tolist() == [[0.0, 0.0, 30.0, 0.0]]


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

def test_rmsnorm_constant_row_closed_form():
    eps = 1e-6
    for c in (0.5, -3.0, 1e-4, 200.0):
        x = bf16_of(np.full((1, 64), c, np.float32))
        w = bf16_of(np.linspace(0.5, 1.5, 64).astype(np.float32))
        y = oracle.rmsnorm(x, w, eps)
        cv = bf16_bits_to_f64(x)[0, 0]
        expect = np.sign(cv) * abs(cv) / math.sqrt(cv * cv + eps) * bf16_bits_to_f64(w)
        ref = np.array([bf16_nearest_bruteforce(v) for v in expect], dtype=np.uint16)
        assert np.array_equal(y[0], ref)


def test_rmsnorm_unit_weight_gives_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(6)
    x = bf16_of(rng.standard_normal((4, 5120)).astype(np.float32) * 7)
    w = bf16_of(np.ones(5120, np.float32))
    y = bf16_bits_to_f64(oracle.rmsnorm(x, w, 1e-6))
    np.testing.assert_allclose(np.sqrt((y ** 2).mean(axis=1)), 1.0, rtol=2e-3)
    x2 = bf16_of(bf16_bits_to_f64(x).astype(np.float32) * 4)   # exact power-of-two scaling
    y2 = bf16_bits_to_f64(oracle.rmsnorm(x2, w, 1e-6))
    assert np.max(np.abs(y2 - y)) <= 2.0 ** -7 * np.max(np.abs(y))
    # each row normalised by its own statistics
    ya = bf16_bits_to_f64(oracle.rmsnorm(x[1:2], w, 1e-6))
    assert np.array_equal(ya[0], y[1])


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

def test_rope_position_zero_is_identity():
    rng = np.random.default_rng(7)
    x = bf16_of(rng.standard_normal((3, 4, 64)).astype(np.float32))
    y = oracle.rope(x, np.zeros(3, np.int32), 1e6)
    assert np.array_equal(x, y)


def test_rope_frequencies_and_pairing_closed_form():
    theta = 1e6
    # D = 4: pairs (0, 2) with inv_freq 1 and (1, 3) with inv_freq theta^-1/2 = 1e-3
    x = np.zeros((2, 1, 4), np.float32)
    x[0, 0, 0] = 1.0      # first pair, position 1 -> (cos 1, sin 1) at indices 0, 2
    x[1, 0, 1] = 1.0      # second pair, position 1000 -> angle 1 at indices 1, 3
    y = bf16_bits_to_f64(oracle.rope(bf16_of(x), np.array([1, 1000], np.int32), theta))
    c, s = math.cos(1.0), math.sin(1.0)
    tol = 2.0 ** -8
    np.testing.assert_allclose(y[0, 0], [c, 0, s, 0], atol=tol)
    np.testing.assert_allclose(y[1, 0], [0, c, 0, s], atol=tol)
    # rotating the second element of a pair: (x1, x2) = (0, 1) -> (-sin, cos)
    x = np.zeros((1, 1, 4), np.float32)
    x[0, 0, 2] = 1.0
    y = bf16_bits_to_f64(oracle.rope(bf16_of(x), np.array([1], np.int32), theta))
    np.testing.assert_allclose(y[0, 0], [-s, 0, c, 0], atol=tol)


def test_rope_preserves_norm_and_relative_position():
    rng = np.random.default_rng(8)
    D = 128
    q = bf16_of(rng.standard_normal((1, 1, D)).astype(np.float32))
    k = bf16_of(rng.standard_normal((1, 1, D)).astype(np.float32))
    qv = bf16_bits_to_f64(q)
    for p in (1, 17, 255, 4095):
        y = bf16_bits_to_f64(oracle.rope(q, np.array([p], np.int32), 1e6))
        np.testing.assert_allclose(np.linalg.norm(y), np.linalg.norm(qv), rtol=4e-3)

    def dot(m, n):
        a = bf16_bits_to_f64(oracle.rope(q, np.array([m], np.int32), 1e6))
        b = bf16_bits_to_f64(oracle.rope(k, np.array([n], np.int32), 1e6))
        return float((a * b).sum())
    ref = dot(5, 3)
    for shift in (10, 100, 1000):
        assert abs(dot(5 + shift, 3 + shift) - ref) <= 0.05 * np.linalg.norm(qv) * 1.0 + 0.2


# ---------------------------------------------------------------------------
# KV write and attention
# ---------------------------------------------------------------------------

def test_kv_write_readback_and_skip():
    Hkv, D, page, nblk = 2, 8, 4, 3
    kc = np.zeros((nblk * page, Hkv, D), np.uint16)
    vc = np.zeros_like(kc)
    rng = np.random.default_rng(9)
    k = rng.integers(1, 60000, (3, Hkv, D)).astype(np.uint16)
    v = rng.integers(1, 60000, (3, Hkv, D)).astype(np.uint16)
    rc = oracle.kv_write(k, v, np.array([5, -1, 11], np.int32), kc, vc)
    assert rc == 0
    assert np.array_equal(kc[5], k[0]) and np.array_equal(vc[5], v[0])
    assert np.array_equal(kc[11], k[2]) and np.array_equal(vc[11], v[2])
    untouched = [i for i in range(nblk * page) if i not in (5, 11)]
    assert not kc[untouched].any() and not vc[untouched].any()
    assert oracle.kv_write(k, v, np.array([12, -1, 0], np.int32), kc, vc) == -3


def _contiguous_case(rng, B, Hq, Hkv, D, page, ctx, shuffle_seed=None):
    nb = int(math.ceil(max(ctx) / page))
    phys = B * nb
    perm = np.arange(phys, dtype=np.int32)
    if shuffle_seed is not None:
        perm = np.random.default_rng(shuffle_seed).permutation(phys).astype(np.int32)
    bt = perm.reshape(B, nb)
    kvals = bf16_of(rng.standard_normal((B, nb * page, Hkv, D)).astype(np.float32))
    vvals = bf16_of(rng.standard_normal((B, nb * page, Hkv, D)).astype(np.float32))
    kc = np.zeros((phys * page, Hkv, D), np.uint16)
    vc = np.zeros_like(kc)
    for b in range(B):
        for t in range(nb * page):
            s = bt[b, t // page] * page + t % page
            kc[s] = kvals[b, t]
            vc[s] = vvals[b, t]
    return bt, kc, vc


def test_attention_single_token_returns_v_and_gqa_mapping():
    Hq, Hkv, D, page = 4, 2, 16, 4
    rng = np.random.default_rng(10)
    q = bf16_of(rng.standard_normal((1, Hq, D)).astype(np.float32))
    kc = bf16_of(rng.standard_normal((page, Hkv, D)).astype(np.float32))
    vc = np.zeros((page, Hkv, D), np.uint16)
    vc[0, 0] = bf16_of(np.full(D, 1.0, np.float32))
    vc[0, 1] = bf16_of(np.full(D, 2.0, np.float32))
    out, rc = oracle.paged_attention(q, kc, vc, np.array([[0]], np.int32),
                                     np.array([1], np.int32), page)
    assert rc == 0
    ov = bf16_bits_to_f64(out)
    # query heads 0,1 read KV head 0; heads 2,3 read KV head 1 (contiguous groups)
    assert np.all(ov[0, 0] == 1.0) and np.all(ov[0, 1] == 1.0)
    assert np.all(ov[0, 2] == 2.0) and np.all(ov[0, 3] == 2.0)


def test_attention_scale_and_softmax_closed_form():
    D, page = 16, 4
    a = 3.0
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = a
    kc = np.zeros((page, 1, D), np.float32)
    kc[0, 0, 0] = 1.0                      # s0 = a / sqrt(D), s1 = 0
    vc = np.zeros((page, 1, D), np.float32)
    vc[0, 0, 3] = 1.0
    vc[1, 0, 4] = 1.0
    out, _ = oracle.paged_attention(bf16_of(q), bf16_of(kc), bf16_of(vc),
                                    np.array([[0]], np.int32), np.array([2], np.int32), page)
    p0 = 1.0 / (1.0 + math.exp(-a / math.sqrt(D)))
    ov = bf16_bits_to_f64(out)[0, 0]
    assert abs(ov[3] - p0) <= 2.0 ** -9 and abs(ov[4] - (1 - p0)) <= 2.0 ** -9
    assert ov[0] == 0 and ov[5] == 0


def test_attention_q_zero_is_mean_of_v_and_constant_v():
    rng = np.random.default_rng(11)
    B, Hq, Hkv, D, page = 2, 4, 2, 32, 8
    ctx = [13, 20]
    bt, kc, vc = _contiguous_case(rng, B, Hq, Hkv, D, page, ctx)
    q = np.zeros((B, Hq, D), np.uint16)
    out, _ = oracle.paged_attention(q, kc, vc, bt, np.array(ctx, np.int32), page)
    ov = bf16_bits_to_f64(out)
    for b in range(B):
        for h in range(Hq):
            vs = [bf16_bits_to_f64(vc[bt[b, t // page] * page + t % page, h // 2]) for t in range(ctx[b])]
            np.testing.assert_allclose(ov[b, h], np.mean(vs, axis=0), atol=2.0 ** -8 * 4)
    # constant V: softmax weights sum to one whatever q is
    vconst = np.zeros_like(vc)
    vconst[:] = bf16_of(np.float32(1.5))
    q = bf16_of(rng.standard_normal((B, Hq, D)).astype(np.float32) * 3)
    out, _ = oracle.paged_attention(q, kc, vconst, bt, np.array(ctx, np.int32), page)
    assert np.all(bf16_bits_to_f64(out) == 1.5)


def test_attention_paged_equals_contiguous_and_shuffle_invariant():
    rng = np.random.default_rng(12)
    B, Hq, Hkv, D, page = 3, 8, 2, 64, 16
    ctx = [1, 37, 64]
    bt0, kc0, vc0 = _contiguous_case(np.random.default_rng(13), B, Hq, Hkv, D, page, ctx)
    bt1, kc1, vc1 = _contiguous_case(np.random.default_rng(13), B, Hq, Hkv, D, page, ctx,
                                     shuffle_seed=99)
    assert not np.array_equal(bt0, bt1)
    q = bf16_of(rng.standard_normal((B, Hq, D)).astype(np.float32))
    o0, _ = oracle.paged_attention(q, kc0, vc0, bt0, np.array(ctx, np.int32), page)
    o1, _ = oracle.paged_attention(q, kc1, vc1, bt1, np.array(ctx, np.int32), page)
    assert np.array_equal(o0, o1)
    # contiguous layout (page = whole context, identity table) gives the same result
    big = 64
    kcc = np.zeros((B * big, Hkv, D), np.uint16)
    vcc = np.zeros_like(kcc)
    for b in range(B):
        for t in range(ctx[b]):
            s = bt0[b, t // page] * page + t % page
            kcc[b * big + t] = kc0[s]
            vcc[b * big + t] = vc0[s]
    o2, _ = oracle.paged_attention(q, kcc, vcc, np.arange(B, dtype=np.int32)[:, None],
                                   np.array(ctx, np.int32), big)
    assert np.array_equal(o0, o2)


def test_attention_padded_row_and_bounds():
    rng = np.random.default_rng(14)
    B, Hq, Hkv, D, page = 2, 2, 1, 8, 4
    bt, kc, vc = _contiguous_case(rng, B, Hq, Hkv, D, page, [4, 4])
    q = bf16_of(rng.standard_normal((B, Hq, D)).astype(np.float32))
    out, rc = oracle.paged_attention(q, kc, vc, bt, np.array([0, 4], np.int32), page)
    assert rc == 0 and not out[0].any() and out[1].any()
    bad = bt.copy()
    bad[1, 0] = 99
    out, rc = oracle.paged_attention(q, kc, vc, bad, np.array([0, 4], np.int32), page)
    assert rc == -3 and not out[1].any()


# ---------------------------------------------------------------------------
# INT8 KV variant: INT8 cache rows with FP32 row scales
# ---------------------------------------------------------------------------

def _pow2_rows(rng, shape, e_lo=-6, e_hi=2):
    """BF16 rows (last axis) whose absmax is 127 * 2^e: integer codes in
    [-127, 127] with one +-127 per row, times a power of two per row. Returns
    (bf16 bits, codes int8, scales float32); every value is exact in BF16."""
    codes = rng.integers(-127, 128, shape)
    flat = codes.reshape(-1, shape[-1])
    at = rng.integers(0, shape[-1], flat.shape[0])
    flat[np.arange(flat.shape[0]), at] = rng.choice([-127, 127], flat.shape[0])
    e = rng.integers(e_lo, e_hi + 1, shape[:-1])
    scales = np.ldexp(1.0, e)
    vals = codes * scales[..., None]
    return bf16_of(vals.astype(np.float32)), codes.astype(np.int8), scales.astype(np.float32)


def test_kv_write_i8_quantises_each_head_row_at_its_slot():
    Hkv, D, page, nblk = 2, 16, 4, 3
    rng = np.random.default_rng(30)
    mag = np.array([0.05, 7.0])[None, :, None]          # heads of different size
    k = bf16_of((rng.standard_normal((3, Hkv, D)) * mag).astype(np.float32))
    v = bf16_of((rng.standard_normal((3, Hkv, D)) * mag[:, ::-1]).astype(np.float32))
    k[1, 0] = 0                                          # an all-zero row
    n = nblk * page
    kc = np.full((n, Hkv, D), 5, np.int8)
    vc = np.full((n, Hkv, D), 5, np.int8)
    ks = np.full((n, Hkv), -1.0, np.float32)
    vs = np.full((n, Hkv), -1.0, np.float32)
    rc = oracle.kv_write_i8(k, v, np.array([5, 2, 11], np.int32), kc, vc, ks, vs)
    assert rc == 0
    for t, sl in ((0, 5), (1, 2), (2, 11)):
        for x, c, sc in ((k[t], kc[sl], ks[sl]), (v[t], vc[sl], vs[sl])):
            q, qs = oracle.quant_rows(x)                 # the head rows of one token
            assert np.array_equal(c, q) and np.array_equal(sc, qs)
            xv = bf16_bits_to_f64(x)
            for h in range(Hkv):
                if sc[h] == 0:
                    assert not xv[h].any() and not c[h].any()
                    continue
                # round to nearest: within half a step of the row's scale
                err = np.abs(xv[h] - c[h].astype(np.float64) * float(sc[h]))
                assert err.max() <= 0.5 * float(sc[h]) * (1 + 2.0 ** -20)
                assert np.abs(c[h]).max() == 127
    assert not kc[2, 0].any() and ks[2, 0] == 0          # the zero row (token 1, slot 2)
    untouched = [i for i in range(n) if i not in (2, 5, 11)]
    assert np.all(kc[untouched] == 5) and np.all(ks[untouched] == -1.0)
    assert np.all(vc[untouched] == 5) and np.all(vs[untouched] == -1.0)
    # an out-of-range slot writes nothing for that token and reports -3
    kc2, ks2 = kc.copy(), ks.copy()
    assert oracle.kv_write_i8(k, v, np.array([n, -1, -1], np.int32), kc2, vc.copy(), ks2,
                              vs.copy()) == -3
    assert np.array_equal(kc2, kc) and np.array_equal(ks2, ks)


def test_kv_write_i8_recovers_codes_and_power_of_two_scales_exactly():
    rng = np.random.default_rng(31)
    T, Hkv, D = 6, 3, 32
    k, kcodes, kscales = _pow2_rows(rng, (T, Hkv, D))
    v, vcodes, vscales = _pow2_rows(rng, (T, Hkv, D))
    kc = np.zeros((T, Hkv, D), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros((T, Hkv), np.float32)
    vs = np.zeros_like(ks)
    assert oracle.kv_write_i8(k, v, np.arange(T, dtype=np.int32)[::-1].copy(), kc, vc, ks, vs) == 0
    assert np.array_equal(kc[::-1], kcodes) and np.array_equal(ks[::-1], kscales)
    assert np.array_equal(vc[::-1], vcodes) and np.array_equal(vs[::-1], vscales)


def test_attention_i8_exact_cache_equals_bf16_attention():
    """Rows that INT8 represents exactly reduce the variant to the BF16 form:
    K and V scales differ per token, per head and between K and V, so a
    misplaced or swapped scale, or a missing dequantisation, changes the result."""
    rng = np.random.default_rng(32)
    B, Hq, Hkv, D, page = 3, 8, 2, 64, 16
    ctx = [1, 37, 64]
    nb = 4
    phys = B * nb
    bt = rng.permutation(phys).astype(np.int32).reshape(B, nb)
    kb, kcodes, kscales = _pow2_rows(rng, (phys * page, Hkv, D))
    vb, vcodes, vscales = _pow2_rows(rng, (phys * page, Hkv, D), e_lo=-3, e_hi=5)
    q = bf16_of(rng.standard_normal((B, Hq, D)).astype(np.float32) * 0.1)
    cl = np.array(ctx, np.int32)
    ref, rc0 = oracle.paged_attention(q, kb, vb, bt, cl, page)
    out, rc1 = oracle.paged_attention_i8(q, kcodes, vcodes, kscales, vscales, bt, cl, page)
    assert rc0 == 0 and rc1 == 0
    assert np.array_equal(out, ref)
    # the same cache with K and V scales exchanged is a different cache
    swapped, _ = oracle.paged_attention_i8(q, kcodes, vcodes, vscales, kscales, bt, cl, page)
    assert not np.array_equal(swapped, ref)


def test_attention_i8_single_token_returns_dequantised_v():
    rng = np.random.default_rng(33)
    Hq, Hkv, D, page = 4, 2, 16, 4
    q = bf16_of(rng.standard_normal((1, Hq, D)).astype(np.float32))
    kc = rng.integers(-127, 128, (page, Hkv, D)).astype(np.int8)
    vc = rng.integers(-127, 128, (page, Hkv, D)).astype(np.int8)
    ks = rng.uniform(1e-3, 1e-1, (page, Hkv)).astype(np.float32)
    vs = rng.uniform(1e-3, 1e-1, (page, Hkv)).astype(np.float32)
    out, rc = oracle.paged_attention_i8(q, kc, vc, ks, vs, np.array([[0]], np.int32),
                                        np.array([1], np.int32), page)
    assert rc == 0
    for h in range(Hq):
        kvh = h // 2
        want = oracle.bf16_from_f64(vc[0, kvh].astype(np.float64) * float(vs[0, kvh]))
        assert np.array_equal(out[0, h], want)


def test_attention_i8_padded_row_and_bounds():
    rng = np.random.default_rng(34)
    B, Hq, Hkv, D, page = 2, 2, 1, 8, 4
    bt = np.array([[0], [1]], np.int32)
    kc = rng.integers(-127, 128, (2 * page, Hkv, D)).astype(np.int8)
    vc = rng.integers(-127, 128, (2 * page, Hkv, D)).astype(np.int8)
    ks = np.full((2 * page, Hkv), 0.01, np.float32)
    q = bf16_of(rng.standard_normal((B, Hq, D)).astype(np.float32))
    out, rc = oracle.paged_attention_i8(q, kc, vc, ks, ks, bt, np.array([0, 4], np.int32), page)
    assert rc == 0 and not out[0].any() and out[1].any()
    bad = bt.copy()
    bad[1, 0] = 2
    out, rc = oracle.paged_attention_i8(q, kc, vc, ks, ks, bad, np.array([0, 4], np.int32), page)
    assert rc == -3 and not out[1].any()


# ---------------------------------------------------------------------------
# Gate/Up + SwiGLU
# ---------------------------------------------------------------------------

def test_gate_up_swiglu_closed_forms_and_row_layout():
    I, K = 4, 16
    W = np.zeros((2 * I, K), np.int8)
    xq = np.zeros((1, K), np.int8)
    xq[0, 0] = 1
    g_vals = [0, 1, 40, -40]
    for j in range(I):
        W[j, 0] = g_vals[j]        # gate rows first
        W[I + j, 0] = 2            # up rows after
    s = np.ones(2 * I, np.float32)
    act, acc = oracle.gate_up_swiglu(xq, np.array([1.0], np.float32), W, s)
    assert acc[0].tolist() == g_vals + [2] * I
    av = bf16_bits_to_f64(act)[0]
    expect = [0.0, 2.0 / (1.0 + math.exp(-1.0)), 80.0, 2.0 * -40.0 / (1.0 + math.exp(40.0))]
    for got, e in zip(av, expect):
        assert abs(got - e) <= abs(e) * 2.0 ** -8 + 1e-30, (got, e)


# ---------------------------------------------------------------------------
# Layer wiring
# ---------------------------------------------------------------------------

def _tiny_case(B=1, ctx=(16,), seed=21, padded=()):
    cfg = synth.TINY
    case = synth.decode_layer_case(cfg, B, list(ctx), seed_base=seed, padded_rows=padded)
    return cfg, case


def _run_layer(cfg, case, taps=True, weights=None):
    kc = case["k_cache"].copy()
    vc = case["v_cache"].copy()
    h, t, rc = oracle.decode_layer(weights or case["weights"], cfg, case["hidden"],
                                   case["slot_mapping"], case["block_table"],
                                   case["ctx_lens"], kc, vc, taps=taps)
    return h, t, rc, kc, vc


def test_layer_taps_compose_the_pinned_steps():
    cfg, case = _tiny_case(B=2, ctx=(16, 9))
    h, t, rc, kc, vc = _run_layer(cfg, case)
    assert rc == 0
    w = case["weights"]
    eps, D = cfg["rms_eps"], cfg["head_dim"]
    Hq, Hkv = cfg["num_q_heads"], cfg["num_kv_heads"]
    assert np.array_equal(t["xn"], oracle.rmsnorm(case["hidden"], w["input_norm_w"], eps))
    q, s = oracle.quant_rows(t["xn"])
    assert np.array_equal(t["xq"], q) and np.array_equal(t["xs"], s)
    y, acc = oracle.linear(t["xq"], t["xs"], w["w_qkv"], w["s_qkv"])
    assert np.array_equal(t["qkv"], y)
    assert np.array_equal(t["acc_qkv"], t["xq"].astype(np.int64) @ w["w_qkv"].astype(np.int64).T)
    NQ, NK = Hq * D, Hkv * D
    qh = oracle.rmsnorm(t["qkv"][:, :NQ].reshape(2, Hq, D), w["q_norm_w"], eps)
    kh = oracle.rmsnorm(t["qkv"][:, NQ:NQ + NK].reshape(2, Hkv, D), w["k_norm_w"], eps)
    pos = case["ctx_lens"] - 1
    assert np.array_equal(t["q_rot"], oracle.rope(qh, pos, cfg["rope_theta"]))
    assert np.array_equal(t["k_rot"], oracle.rope(kh, pos, cfg["rope_theta"]))
    # KV landed at each row's slot
    for b in range(2):
        sl = case["slot_mapping"][b]
        assert np.array_equal(kc[sl], t["k_rot"][b])
        assert np.array_equal(vc[sl], t["qkv"][b, NQ + NK:].reshape(Hkv, D))
    att, _ = oracle.paged_attention(t["q_rot"], kc, vc, case["block_table"], case["ctx_lens"],
                                    cfg["page_size"])
    assert np.array_equal(t["attn"], att.reshape(2, NQ))
    aq, as_ = oracle.quant_rows(t["attn"])
    h1, _ = oracle.linear(aq, as_, w["w_o"], w["s_o"], 1, case["hidden"])
    assert np.array_equal(t["h1"], h1)
    hq, hs = oracle.quant_rows(oracle.rmsnorm(h1, w["post_norm_w"], eps))
    act, _ = oracle.gate_up_swiglu(hq, hs, w["w_gate_up"], w["s_gate_up"])
    assert np.array_equal(t["act"], act)
    dq, ds = oracle.quant_rows(act)
    out, _ = oracle.linear(dq, ds, w["w_down"], w["s_down"], 2, h1)
    assert np.array_equal(h, out)


def test_layer_zero_projections_keep_residual():
    cfg, case = _tiny_case()
    w = dict(case["weights"])
    w["w_o"] = np.zeros_like(w["w_o"])
    w["w_down"] = np.zeros_like(w["w_down"])
    h, t, rc, _, _ = _run_layer(cfg, case, weights=w)
    assert rc == 0
    assert np.array_equal(t["h1"], case["hidden"])
    assert np.array_equal(h, case["hidden"])


def test_layer_rows_independent_and_padding():
    cfg, case = _tiny_case(B=3, ctx=(16, 5, 16), padded=(1,))
    h, t, rc, kc, vc = _run_layer(cfg, case)
    assert rc == 0
    assert not t["attn"][1].any()
    for b in (0, 2):
        sub = dict(case)
        sub["hidden"] = case["hidden"][b:b + 1]
        sub["slot_mapping"] = case["slot_mapping"][b:b + 1]
        sub["block_table"] = case["block_table"][b:b + 1]
        sub["ctx_lens"] = case["ctx_lens"][b:b + 1]
        hb, _, rcb, _, _ = _run_layer(cfg, sub, taps=False)
        assert rcb == 0 and np.array_equal(hb[0], h[b])
    # the padded row wrote nothing: only rows 0 and 2 changed the caches
    changed = np.nonzero((kc != case["k_cache"]).any(axis=(1, 2)))[0].tolist()
    assert sorted(changed) == sorted(case["slot_mapping"][[0, 2]].tolist())


def test_layer_first_token_attends_to_itself():
    cfg, case = _tiny_case(ctx=(1,))
    _, t, rc, _, _ = _run_layer(cfg, case)
    assert rc == 0
    D, Hq, Hkv = cfg["head_dim"], cfg["num_q_heads"], cfg["num_kv_heads"]
    NQ, NK = Hq * D, Hkv * D
    v = t["qkv"][0, NQ + NK:].reshape(Hkv, D)
    att = t["attn"][0].reshape(Hq, D)
    for h in range(Hq):
        assert np.array_equal(att[h], v[h // (Hq // Hkv)])


def _i8_history(seed, like):
    return synth.i8_kv_history(seed, like.shape[0], like.shape[1], like.shape[2])


def test_layer_i8kv_shares_the_bf16_steps_and_quantises_the_written_rows():
    cfg, case = _tiny_case(B=2, ctx=(16, 9))
    _, tb, rc0, _, _ = _run_layer(cfg, case)
    kc, ks = _i8_history(35, case["k_cache"])
    vc, vs = _i8_history(36, case["v_cache"])
    kc0, vc0, ks0, vs0 = kc.copy(), vc.copy(), ks.copy(), vs.copy()
    w = case["weights"]
    h, t, rc = oracle.decode_layer(w, cfg, case["hidden"], case["slot_mapping"],
                                   case["block_table"], case["ctx_lens"], kc, vc, taps=True,
                                   k_scale=ks, v_scale=vs)
    assert rc0 == 0 and rc == 0
    # everything before the cache write is the BF16-cache layer's
    for name in ("xn", "xq", "xs", "acc_qkv", "qkv", "q_rot", "k_rot"):
        assert np.array_equal(t[name], tb[name]), name
    Hq, Hkv, D = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    NQ, NK = Hq * D, Hkv * D
    written = set()
    for b in range(2):
        sl = case["slot_mapping"][b]
        written.add(int(sl))
        q, qs = oracle.quant_rows(t["k_rot"][b])
        assert np.array_equal(kc[sl], q) and np.array_equal(ks[sl], qs)
        q, qs = oracle.quant_rows(t["qkv"][b, NQ + NK:].reshape(Hkv, D))
        assert np.array_equal(vc[sl], q) and np.array_equal(vs[sl], qs)
    rest = [i for i in range(kc.shape[0]) if i not in written]
    assert np.array_equal(kc[rest], kc0[rest]) and np.array_equal(ks[rest], ks0[rest])
    assert np.array_equal(vc[rest], vc0[rest]) and np.array_equal(vs[rest], vs0[rest])
    # attention reads the INT8 cache; the steps after it are the pinned ones
    att, _ = oracle.paged_attention_i8(t["q_rot"], kc, vc, ks, vs, case["block_table"],
                                       case["ctx_lens"], cfg["page_size"])
    assert np.array_equal(t["attn"], att.reshape(2, NQ))
    aq, as_ = oracle.quant_rows(t["attn"])
    h1, _ = oracle.linear(aq, as_, w["w_o"], w["s_o"], 1, case["hidden"])
    assert np.array_equal(t["h1"], h1)
    hq, hs = oracle.quant_rows(oracle.rmsnorm(h1, w["post_norm_w"], cfg["rms_eps"]))
    act, _ = oracle.gate_up_swiglu(hq, hs, w["w_gate_up"], w["s_gate_up"])
    dq, ds = oracle.quant_rows(act)
    out, _ = oracle.linear(dq, ds, w["w_down"], w["s_down"], 2, h1)
    assert np.array_equal(h, out)


def test_layer_i8kv_first_token_attends_to_its_dequantised_v():
    cfg, case = _tiny_case(ctx=(1,))
    kc, ks = _i8_history(37, case["k_cache"])
    vc, vs = _i8_history(38, case["v_cache"])
    _, t, rc = oracle.decode_layer(case["weights"], cfg, case["hidden"], case["slot_mapping"],
                                   case["block_table"], case["ctx_lens"], kc, vc, taps=True,
                                   k_scale=ks, v_scale=vs)
    assert rc == 0
    Hq, Hkv, D = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    sl = case["slot_mapping"][0]
    att = t["attn"][0].reshape(Hq, D)
    for h in range(Hq):
        kvh = h // (Hq // Hkv)
        want = oracle.bf16_from_f64(vc[sl, kvh].astype(np.float64) * float(vs[sl, kvh]))
        assert np.array_equal(att[h], want)


# ---------------------------------------------------------------------------
# BF16 (unquantised) layer variant
# ---------------------------------------------------------------------------

def test_linear_bf16_is_the_exact_sum_rounded_once():
    rng = np.random.default_rng(40)
    M, K, N = 2, 40, 5
    x = bf16_of(rng.standard_normal((M, K)).astype(np.float32))
    W = bf16_of((rng.standard_normal((N, K)) * 0.05).astype(np.float32))
    res = bf16_of((rng.standard_normal((M, N)) * 3).astype(np.float32))
    xv, Wv, rv = bf16_bits_to_f64(x), bf16_bits_to_f64(W), bf16_bits_to_f64(res)
    for residual in (None, res):
        y = oracle.linear_bf16(x, W, residual)
        for m in range(M):
            for n in range(N):
                exact = sum(Fraction(float(xv[m, k])) * Fraction(float(Wv[n, k]))
                            for k in range(K))
                if residual is not None:
                    exact += Fraction(float(rv[m, n]))
                assert int(y[m, n]) == bf16_nearest_bruteforce(float(exact)), (m, n)
    # one narrowing of (sum + residual): 1 + 2^-8 + 2^-20 rounds up to 1 + 2^-7,
    # while narrowing the sum first (to 2^-8) would leave a tie that rounds to 1
    x1 = bf16_of(np.array([[1.0, 1.0]], np.float32))
    W1 = bf16_of(np.array([[2.0 ** -8, 2.0 ** -20]], np.float32))
    y1 = oracle.linear_bf16(x1, W1, bf16_of(np.array([[1.0]], np.float32)))
    assert bf16_bits_to_f64(y1)[0, 0] == 1.0 + 2.0 ** -7


def test_linear_bf16_on_scaled_codes_equals_the_a8w8_projection():
    """x = q 2^a and W = c 2^b (exact in BF16): the A8W8 projection of (q, 2^a,
    c, 2^b) is bf16(acc 2^(a+b)) exactly while |acc| < 2^24, and so must be the
    real-valued BF16 projection; a transposed or misrouted operand breaks it."""
    rng = np.random.default_rng(41)
    M, K, N = 3, 256, 24
    q = rng.integers(-127, 128, (M, K)).astype(np.int8)
    c = rng.integers(-127, 128, (N, K)).astype(np.int8)
    a = rng.integers(-9, -3, M)
    b = rng.integers(-12, -6, N)
    x = bf16_of((q * np.ldexp(1.0, a)[:, None]).astype(np.float32))
    W = bf16_of((c * np.ldexp(1.0, b)[:, None]).astype(np.float32))
    y8, acc = oracle.linear(q, np.ldexp(1.0, a).astype(np.float32), c,
                            np.ldexp(1.0, b).astype(np.float32))
    assert np.abs(acc).max() < 2 ** 24
    assert np.array_equal(oracle.linear_bf16(x, W), y8)


def test_gate_up_swiglu_bf16_bruteforce():
    """g and u are the exact sums, not narrowed; act = bf16(silu(g) u) once."""
    rng = np.random.default_rng(43)
    M, K, I = 2, 24, 6
    x = bf16_of(rng.standard_normal((M, K)).astype(np.float32))
    W = bf16_of((rng.standard_normal((2 * I, K)) * 0.3).astype(np.float32))
    act = oracle.gate_up_swiglu_bf16(x, W)
    xv, Wv = bf16_bits_to_f64(x), bf16_bits_to_f64(W)
    for m in range(M):
        for j in range(I):
            g = float(sum(Fraction(float(xv[m, k])) * Fraction(float(Wv[j, k])) for k in range(K)))
            u = float(sum(Fraction(float(xv[m, k])) * Fraction(float(Wv[I + j, k]))
                          for k in range(K)))
            assert int(act[m, j]) == bf16_nearest_bruteforce(g / (1.0 + math.exp(-g)) * u), (m, j)


def test_gate_up_swiglu_bf16_closed_forms_and_row_layout():
    I, K = 4, 8
    x = np.zeros((1, K), np.float32)
    x[0, 0] = 1.0
    g_vals = [0.0, 1.0, 40.0, -40.0]
    u_vals = [5.0, 2.0, 1.0, 1.0]
    W = np.zeros((2 * I, K), np.float32)
    for j in range(I):
        W[j, 0] = g_vals[j]            # gate rows first
        W[I + j, 0] = u_vals[j]        # then up rows
    bits = oracle.gate_up_swiglu_bf16(bf16_of(x), bf16_of(W))[0]
    act = bf16_bits_to_f64(bits)
    assert act[0] == 0.0
    assert int(bits[1]) == bf16_nearest_bruteforce(2.0 / (1.0 + math.exp(-1.0)))
    assert act[2] == 40.0                                  # silu(40) = 40 to BF16
    assert int(bits[3]) == bf16_nearest_bruteforce(-40.0 / (1.0 + math.exp(40.0)))
    assert act[3] < 0


def _bf16_case(B=2, ctx=(16, 9), seed=42):
    cfg = synth.TINY
    case = synth.decode_layer_case(cfg, B, list(ctx), seed_base=seed)
    case["weights"] = synth.bf16_layer_weights(cfg, seed)
    return cfg, case


def _run_bf16_layer(cfg, case, weights=None):
    kc, vc = case["k_cache"].copy(), case["v_cache"].copy()
    h, t, rc = oracle.decode_layer_bf16(weights or case["weights"], cfg, case["hidden"],
                                        case["slot_mapping"], case["block_table"],
                                        case["ctx_lens"], kc, vc, taps=True)
    return h, t, rc, kc, vc


def test_layer_bf16_taps_compose_the_pinned_steps():
    cfg, case = _bf16_case()
    h, t, rc, kc, vc = _run_bf16_layer(cfg, case)
    assert rc == 0
    w = case["weights"]
    eps, D = cfg["rms_eps"], cfg["head_dim"]
    Hq, Hkv = cfg["num_q_heads"], cfg["num_kv_heads"]
    NQ, NK = Hq * D, Hkv * D
    assert np.array_equal(t["xn"], oracle.rmsnorm(case["hidden"], w["input_norm_w"], eps))
    assert np.array_equal(t["qkv"], oracle.linear_bf16(t["xn"], w["w_qkv"]))
    qh = oracle.rmsnorm(t["qkv"][:, :NQ].reshape(2, Hq, D), w["q_norm_w"], eps)
    kh = oracle.rmsnorm(t["qkv"][:, NQ:NQ + NK].reshape(2, Hkv, D), w["k_norm_w"], eps)
    pos = case["ctx_lens"] - 1
    assert np.array_equal(t["q_rot"], oracle.rope(qh, pos, cfg["rope_theta"]))
    assert np.array_equal(t["k_rot"], oracle.rope(kh, pos, cfg["rope_theta"]))
    for b in range(2):
        sl = case["slot_mapping"][b]
        assert np.array_equal(kc[sl], t["k_rot"][b])
        assert np.array_equal(vc[sl], t["qkv"][b, NQ + NK:].reshape(Hkv, D))
    att, _ = oracle.paged_attention(t["q_rot"], kc, vc, case["block_table"], case["ctx_lens"],
                                    cfg["page_size"])
    assert np.array_equal(t["attn"], att.reshape(2, NQ))
    h1 = oracle.linear_bf16(t["attn"], w["w_o"], case["hidden"])
    assert np.array_equal(t["h1"], h1)
    hn = oracle.rmsnorm(h1, w["post_norm_w"], eps)
    assert np.array_equal(t["hn"], hn)
    act = oracle.gate_up_swiglu_bf16(hn, w["w_gate_up"])
    assert np.array_equal(t["act"], act)
    assert np.array_equal(h, oracle.linear_bf16(act, w["w_down"], h1))


def test_layer_bf16_zero_projections_keep_residual_and_first_token_attends_to_itself():
    cfg, case = _bf16_case(B=1, ctx=(1,))
    w = dict(case["weights"])
    w["w_o"] = np.zeros_like(w["w_o"])
    w["w_down"] = np.zeros_like(w["w_down"])
    h, t, rc, _, _ = _run_bf16_layer(cfg, case, weights=w)
    assert rc == 0
    assert np.array_equal(t["h1"], case["hidden"]) and np.array_equal(h, case["hidden"])
    Hq, Hkv, D = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    v = t["qkv"][0, (Hq + Hkv) * D:].reshape(Hkv, D)
    att = t["attn"][0].reshape(Hq, D)
    for h_ in range(Hq):
        assert np.array_equal(att[h_], v[h_ // (Hq // Hkv)])


# ---------------------------------------------------------------------------
# Step
# ---------------------------------------------------------------------------

def test_argmax_lowest_index_on_ties():
    l = np.array([[1.0, 3.0, 3.0, -1.0], [5.0, 5.0, 5.0, 5.0]])
    assert oracle.argmax_f64(l).tolist() == [1, 0]
    assert oracle.argmax_f32(l.astype(np.float32)).tolist() == [1, 0]
    rng = np.random.default_rng(15)
    x = rng.standard_normal((4, 1000))
    assert np.array_equal(oracle.argmax_f64(x), x.argmax(axis=1))


def test_lm_head_bruteforce():
    rng = np.random.default_rng(16)
    hn = bf16_of(rng.standard_normal((2, 64)).astype(np.float32))
    W = bf16_of(rng.standard_normal((300, 64)).astype(np.float32) * 0.02)
    got = oracle.lm_head(hn, W)
    ref = bf16_bits_to_f64(hn) @ bf16_bits_to_f64(W).T
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_step_composes_embed_layers_norm_head():
    cfg = dict(synth.TINY, num_layers=2, vocab=97)
    model = synth.model_weights_host(cfg, 31)
    B, page = 2, cfg["page_size"]
    ctx = np.array([3, 7], np.int32)
    bt, nblk = synth.paged_layout(32, ctx, page, spare_blocks=1)
    slots = synth.slots_for(bt, ctx - 1, page)
    Hkv, D = cfg["num_kv_heads"], cfg["head_dim"]
    kcs = [synth.kv_cache(40 + l, nblk, page, Hkv, D, bt, ctx - 1) for l in range(2)]
    vcs = [synth.kv_cache(50 + l, nblk, page, Hkv, D, bt, ctx - 1) for l in range(2)]
    tok = np.array([5, 96], np.int32)
    kc2 = [c.copy() for c in kcs]
    vc2 = [c.copy() for c in vcs]
    nxt, fh, logits, rc = oracle.decode_step(model, cfg, tok, slots, bt, ctx, kc2, vc2,
                                             want_logits=True)
    assert rc == 0
    h = model["embed"][tok]
    for l in range(2):
        kc = kcs[l].copy()
        vc = vcs[l].copy()
        h, _, r, = oracle.decode_layer(model["layers"][l], cfg, h, slots, bt, ctx, kc, vc)[:3]
        assert r == 0
        assert np.array_equal(kc, kc2[l]) and np.array_equal(vc, vc2[l])
    hn = oracle.rmsnorm(h, model["final_norm_w"], cfg["rms_eps"])
    assert np.array_equal(fh, hn)
    ref = bf16_bits_to_f64(hn) @ bf16_bits_to_f64(model["lm_head"]).T
    np.testing.assert_allclose(logits, ref, rtol=1e-12, atol=1e-12)
    assert np.array_equal(nxt, ref.argmax(axis=1))
    # out-of-range token id is reported
    _, _, _, rc = oracle.decode_step(model, cfg, np.array([5, 97], np.int32), slots, bt, ctx,
                                     [c.copy() for c in kcs], [c.copy() for c in vcs])
    assert rc == -3


def test_prompt_through_the_step_equals_decoding_it_token_by_token():
    # the first generated token of a prompt (time to first token): the step
    # over all prompt rows at once (each at its own position, causal) gives
    # every row the next token and final hidden state of decoding the prompt
    # one token at a time; the last row's token is the first generated one
    cfg = dict(synth.TINY, num_layers=2, vocab=97)
    model = synth.model_weights_host(cfg, 41)
    page, P = cfg["page_size"], 21
    Hkv, D = cfg["num_kv_heads"], cfg["head_dim"]
    bt_seq, nblk = synth.paged_layout(42, [P + 1], page, spare_blocks=1)
    pos = np.arange(P)
    bt = np.repeat(bt_seq, P, axis=0).astype(np.int32)
    ctx = (pos + 1).astype(np.int32)
    slots = synth.slots_for(bt, pos, page)
    tok = synth.prompt_ids(43, P, cfg["vocab"])
    empty = lambda: [np.zeros((nblk * page, Hkv, D), np.uint16) for _ in range(2)]
    kc1, vc1 = empty(), empty()
    nxt, fh, _, rc = oracle.decode_step(model, cfg, tok, slots, bt, ctx, kc1, vc1)
    assert rc == 0
    kc2, vc2 = empty(), empty()
    for i in range(P):
        r = slice(i, i + 1)
        n1, f1, _, rc = oracle.decode_step(model, cfg, tok[r], slots[r], bt[r], ctx[r], kc2, vc2)
        assert rc == 0
        assert n1[0] == nxt[i] and np.array_equal(f1[0], fh[i])
    assert all(np.array_equal(a, b) for a, b in zip(kc1 + vc1, kc2 + vc2))


def test_prefill_chunk_equals_sequential_decode():
    # a prefill chunk (all rows through the layer at once, each at its own
    # position) must equal decoding the rows one position at a time: same
    # outputs, same caches -- the causal reading of the prefill chunk
    cfg = synth.TINY
    case = synth.prefill_case(cfg, seq_lens=[5, 7], prior_ctx=[3, 0], seed_base=31)
    w = case["weights"]
    kc1, vc1 = case["k_cache"].copy(), case["v_cache"].copy()
    out, _, rc = oracle.prefill_layer(w, cfg, case["hidden"], case["slot_mapping"],
                                      case["block_table"], case["ctx_lens"], kc1, vc1)
    assert rc == 0
    kc2, vc2 = case["k_cache"].copy(), case["v_cache"].copy()
    seq_of = np.repeat(np.arange(2), case["seq_lens"])
    idx = np.arange(len(seq_of)) - np.concatenate([[0], np.cumsum(case["seq_lens"])[:-1]])[seq_of]
    seq_out = np.empty_like(case["hidden"])
    for i in range(int(case["seq_lens"].max())):
        rows = np.nonzero(idx == i)[0]
        h, _, rc = oracle.decode_layer(w, cfg, case["hidden"][rows], case["slot_mapping"][rows],
                                       case["block_table"][rows], case["ctx_lens"][rows], kc2, vc2)
        assert rc == 0
        seq_out[rows] = h
    assert np.array_equal(out, seq_out)
    assert np.array_equal(kc1, kc2) and np.array_equal(vc1, vc2)
    # and a row's output does depend on the earlier rows of its sequence
    h_alone, _, _ = oracle.decode_layer(w, cfg, case["hidden"][4:5], case["slot_mapping"][4:5],
                                        case["block_table"][4:5], case["ctx_lens"][4:5],
                                        case["k_cache"].copy(), case["v_cache"].copy())
    assert not np.array_equal(h_alone[0], out[4])


def test_prefill_chunk_over_int8_cache_equals_sequential_decode():
    # the same causal reading over the INT8 KV cache: every row's K/V is
    # quantised into its slot before any row attends
    cfg = synth.TINY
    case = synth.prefill_case(cfg, seq_lens=[4, 6], prior_ctx=[5, 0], seed_base=33)
    w = case["weights"]
    n, Hkv, D = case["k_cache"].shape
    kc0, ks0 = synth.i8_kv_history(34, n, Hkv, D)
    vc0, vs0 = synth.i8_kv_history(35, n, Hkv, D)
    c1 = [a.copy() for a in (kc0, vc0, ks0, vs0)]
    out, _, rc = oracle.prefill_layer(w, cfg, case["hidden"], case["slot_mapping"],
                                      case["block_table"], case["ctx_lens"], c1[0], c1[1],
                                      k_scale=c1[2], v_scale=c1[3])
    assert rc == 0
    c2 = [a.copy() for a in (kc0, vc0, ks0, vs0)]
    seq_of = np.repeat(np.arange(2), case["seq_lens"])
    idx = np.arange(len(seq_of)) - np.concatenate([[0], np.cumsum(case["seq_lens"])[:-1]])[seq_of]
    seq_out = np.empty_like(case["hidden"])
    for i in range(int(case["seq_lens"].max())):
        rows = np.nonzero(idx == i)[0]
        h, _, rc = oracle.decode_layer(w, cfg, case["hidden"][rows], case["slot_mapping"][rows],
                                       case["block_table"][rows], case["ctx_lens"][rows], c2[0],
                                       c2[1], k_scale=c2[2], v_scale=c2[3])
        assert rc == 0
        seq_out[rows] = h
    assert np.array_equal(out, seq_out)
    assert all(np.array_equal(a, b) for a, b in zip(c1, c2))
    # the chunk's slots hold codes and scales now, and only those changed
    sl = case["slot_mapping"]
    rest = np.setdiff1d(np.arange(n), sl)
    assert np.array_equal(c1[0][rest], kc0[rest]) and np.array_equal(c1[2][rest], ks0[rest])
    assert not np.array_equal(c1[2][sl], ks0[sl])


# ---------------------------------------------------------------------------
# Sampling beyond greedy (oracle/sampling.py)
# ---------------------------------------------------------------------------

from oracle import sampling  # noqa: E402


def test_philox_known_answer_vectors():
    """The published known-answer vectors of Philox4x32-10
    (tests/golden/philox4x32_10_kat.txt): a wrong multiplier, Weyl constant,
    word permutation or round count changes every output word."""
    rows = list(_golden_rows("philox4x32_10_kat.txt"))
    assert len(rows) == 3
    for ctr, key, want in rows:
        c = [np.array([int(w, 16)], np.uint64) for w in ctr.split()]
        k = [int(w, 16) for w in key.split()]
        got = sampling.philox4x32_10(*c, *k)
        assert [int(g[0]) for g in got] == [int(w, 16) for w in want.split()]


def test_philox_is_a_deterministic_bijection_with_uniform_words():
    n = 1 << 16
    i = np.arange(n, dtype=np.uint64)
    z = np.zeros(n, np.uint64)
    w = sampling.philox4x32_10(i, z, z, z, 7, 9)
    w2 = sampling.philox4x32_10(i, z, z, z, 7, 9)
    assert all(np.array_equal(a, b) for a, b in zip(w, w2))
    # a bijection of the 128-bit counter for a fixed key: distinct counters,
    # distinct outputs (checked on the full 128-bit words)
    packed = set(zip(*(x.tolist() for x in w)))
    assert len(packed) == n
    # another key changes every output word
    v = sampling.philox4x32_10(i, z, z, z, 8, 9)
    assert (w[0] != v[0]).mean() > 0.99
    # each word uniform over 32 bits: 16-bin chi-square and bit balance
    for x in w:
        counts = np.bincount((x >> np.uint64(28)).astype(np.int64), minlength=16)
        chi2 = ((counts - n / 16) ** 2 / (n / 16)).sum()
        assert chi2 < 60, chi2           # 15 degrees of freedom: p ~ 1e-7 at 60
        bits = np.unpackbits(x.astype(np.uint32).view(np.uint8)).mean()
        assert abs(bits - 0.5) < 0.005


def test_uniforms_open_interval_and_stream_independence():
    u = sampling.uniforms(100_000, 3, seed=12345, step=7)
    assert u.min() > 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 0.005
    u2 = sampling.uniforms(100_000, 4, seed=12345, step=7)
    u3 = sampling.uniforms(100_000, 3, seed=12345, step=8)
    assert abs(np.corrcoef(u, u2)[0, 1]) < 0.01 and abs(np.corrcoef(u, u3)[0, 1]) < 0.01


def test_sampling_greedy_limits():
    rng = np.random.default_rng(5)
    logits = rng.normal(size=(3, 1000)).astype(np.float32)
    logits[1, 17] = logits[1].max()          # a tie: lowest index wins
    am = np.array([np.argmax(r) for r in logits])
    assert am[1] == 17
    assert np.array_equal(sampling.sample_rows(logits, 0.0, 1.0, 1, 0), am)
    tied = set(np.nonzero(logits[1] == logits[1].max())[0].tolist())
    assert len(tied) == 2
    seen = set()
    for s in range(40):
        # a tiny nucleus holds the maximum alone (both tied maxima in row 1,
        # each drawn with probability 1/2); a tiny temperature likewise
        for x in (sampling.sample_rows(logits, 1.0, 1e-9, s, s),
                  sampling.sample_rows(logits, 1e-6, 1.0, s, s)):
            assert x[0] == am[0] and x[2] == am[2] and x[1] in tied
            seen.add(int(x[1]))
    assert seen == tied


def test_sampling_distribution_is_the_softmax():
    logits = np.array([[1.0, 0.0, -1.0, 2.0, 0.5, -3.0]], np.float32)
    T = 0.8
    p = np.exp(logits[0] / T) / np.exp(logits[0] / T).sum()
    n = 30_000
    draws = np.array([sampling.sample_rows(logits, T, 1.0, 99, s)[0] for s in range(n)])
    freq = np.bincount(draws, minlength=6) / n
    sigma = np.sqrt(p * (1 - p) / n)
    assert (np.abs(freq - p) < 5 * sigma + 1e-4).all(), (freq, p)


def test_sampling_nucleus_renormalises():
    # probabilities 0.5, 0.3, 0.1, 0.05, 0.05: top_p 0.75 keeps {0, 1}
    p = np.array([0.5, 0.3, 0.1, 0.05, 0.05])
    logits = np.log(p)[None, :].astype(np.float32)
    keep = sampling.nucleus(np.log(p) - np.log(p).max(), 0.75)
    assert keep.tolist() == [True, True, False, False, False]
    # the boundary tie is kept whole: top_p 0.92 reaches into the 0.05 pair
    assert sampling.nucleus(np.log(p) - np.log(p).max(), 0.92).tolist() == [True] * 5
    n = 20_000
    draws = np.array([sampling.sample_rows(logits, 1.0, 0.75, 3, s)[0] for s in range(n)])
    freq = np.bincount(draws, minlength=5) / n
    assert freq[2:].sum() == 0
    assert abs(freq[0] - 0.625) < 5 * np.sqrt(0.625 * 0.375 / n)
