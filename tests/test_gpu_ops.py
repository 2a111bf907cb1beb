"""GPU parity of the single operations, through the C ABI, against the oracle.

Integer work (INT8 codes, FP32 scales from the fixed formula, INT32
accumulators, the FP32 dequantisation narrowed to BF16) must match bit for bit
on identical inputs; floating-point stages are held to stated tolerances.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from gpu_util import bf16_close, bf16_to_f64, bf16_ulp_diff, rel_l2, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def a8w8():
    import w8a8_quantized_decode_gb300 as m
    m.build()
    import torch
    torch.cuda.init()
    return m


def _bf16_rows(seed, rows, cols, scale=1.0):
    x = synth.bf16_normal(seed, (rows, cols))
    if scale != 1.0:
        x = synth.bf16_trunc(bf16_to_f64(x).astype(np.float32) * np.float32(scale))
    return x


# ---------------------------------------------------------------------------
# quantisation
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rows,cols", [(1, 5120), (16, 17408), (3, 256), (5, 8), (7, 5128)])
def test_quant_rows_bit_exact(a8w8, rows, cols):
    x = _bf16_rows(rows * 7 + cols, rows, cols, scale=3.0)
    x[0, : min(cols, 8)] = 0          # partial zeros
    if rows > 2:
        x[2] = 0                       # an all-zero row: s = 0, q = 0
    q, s = a8w8.a8w8_quant_rows(to_dev(x))
    oq, os_ = oracle.quant_rows(x)
    assert np.array_equal(to_host(s), os_)
    assert np.array_equal(to_host(q), oq)


def test_quant_rows_golden_ties(a8w8):
    # the hand-derived rows of tests/golden/quant_cases.txt, zero padded to 8 columns
    import os
    rows = []
    with open(os.path.join(os.path.dirname(__file__), "golden", "quant_cases.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                xs = [float(v) for v in line.split("|")[0].split()]
                rows.append(xs + [0.0] * (16 - len(xs)))
    x = synth.bf16_trunc(np.array(rows, np.float32))
    q, s = a8w8.a8w8_quant_rows(to_dev(x))
    oq, os_ = oracle.quant_rows(x)
    assert np.array_equal(to_host(q), oq) and np.array_equal(to_host(s), os_)


# ---------------------------------------------------------------------------
# A8W8 projections
# ---------------------------------------------------------------------------

LINEAR_CASES = [
    # M, K, N, k_splits, residual
    (1, 5120, 7168, 1, False),     # QKV
    (1, 5120, 5120, 1, True),      # O + residual
    (1, 17408, 5120, 2, True),     # down, two-way split-K + residual
    (3, 256, 40, 1, False),        # ragged: K below one 512-byte unit, N below the SM count
    (5, 512, 333, 2, True),
    (8, 5120, 1000, 1, True),
    (16, 17408, 300, 2, True),     # batch tiles of 4
    (11, 4128, 97, 2, False),      # K not a multiple of 512
    # tensor-core form (3..16 rows per launch)
    (16, 5120, 7168, 1, False),    # QKV at batch 16
    (13, 17408, 5120, 2, True),    # down at batch 13: split halves of 136 steps
    (17, 5120, 5120, 1, True),     # two launches (16 + 1 rows)
    (4, 64, 9, 1, True),           # one K step, fewer rows than one 8-row group
]


@pytest.mark.parametrize("M,K,N,ks,with_res", LINEAR_CASES)
def test_linear_bit_exact(a8w8, M, K, N, ks, with_res):
    seed = M * 1000 + K + N
    xq = synth.int8_uniform(seed, (M, K))
    xs = np.random.default_rng(seed).uniform(1e-3, 5e-2, M).astype(np.float32)
    W = synth.int8_uniform(seed + 1, (N, K))
    ws = synth.scales_uniform(seed + 2, N)
    res = _bf16_rows(seed + 3, M, N, scale=20.0) if with_res else None
    y, acc = a8w8.a8w8_linear(to_dev(xq), to_dev(xs), to_dev(W), to_dev(ws), ks,
                              None if res is None else to_dev(res), acc_out=True)
    oy, oacc = oracle.linear(xq, xs, W, ws, ks, res)
    assert np.array_equal(to_host(acc), oacc)
    assert np.array_equal(to_host(y), oy)


def test_linear_residual_in_place(a8w8):
    M, K, N = 2, 5120, 5120
    xq = synth.int8_uniform(1, (M, K))
    xs = np.array([0.01, 0.02], np.float32)
    W = synth.int8_uniform(2, (N, K))
    ws = synth.scales_uniform(3, N)
    h = _bf16_rows(4, M, N, 30.0)
    hd = to_dev(h)
    a8w8.a8w8_linear(to_dev(xq), to_dev(xs), to_dev(W), to_dev(ws), 1, hd, out=hd)
    oy, _ = oracle.linear(xq, xs, W, ws, 1, h)
    assert np.array_equal(to_host(hd), oy)


@pytest.mark.parametrize("M,xv,wv", [(1, 127, 127), (16, 127, 127), (16, -128, -128)])
def test_linear_extreme_values_no_overflow(a8w8, M, xv, wv):
    # the largest products over K = 17408 (|sum| < 2^31); with M >= 3 the
    # tensor-core form (INT8 MMA, INT32 accumulators) runs
    K, N = 17408, 160
    xq = np.full((M, K), xv, np.int8)
    W = np.full((N, K), -wv, np.int8) if wv == 127 else np.full((N, K), wv, np.int8)
    W[::2] = wv
    xs = np.ones(M, np.float32)
    y, acc = a8w8.a8w8_linear(to_dev(xq), to_dev(xs), to_dev(W),
                              to_dev(np.full(N, 1e-6, np.float32)), 2, acc_out=True)
    oy, oacc = oracle.linear(xq, xs, W, np.full(N, 1e-6, np.float32), 2)
    assert np.array_equal(to_host(acc), oacc)
    assert np.array_equal(to_host(y), oy)


@pytest.mark.parametrize("M,K,I", [(1, 5120, 17408), (4, 256, 512), (9, 5120, 700),
                                   (16, 256, 17408), (16, 5120, 2000)])
def test_gate_up_swiglu(a8w8, M, K, I):
    seed = M + K + I
    xq = synth.int8_uniform(seed, (M, K))
    xs = np.random.default_rng(seed).uniform(1e-3, 5e-2, M).astype(np.float32)
    W = synth.int8_uniform(seed + 1, (2 * I, K))
    s = synth.scales_uniform(seed + 2, 2 * I)
    act, acc = a8w8.a8w8_gate_up_swiglu(to_dev(xq), to_dev(xs), to_dev(W), to_dev(s), acc_out=True)
    oact, oacc = oracle.gate_up_swiglu(xq, xs, W, s)
    assert np.array_equal(to_host(acc), oacc)
    # silu(g) * u in two-float on the GPU and in double in the oracle: one
    # BF16 unit in the last place apart at most (measured against the tensor's
    # scale for values near zero), and 99.9% identical
    g = to_host(act)
    assert bf16_close(g, oact, 1, 1e-3).all()
    assert (bf16_ulp_diff(g, oact) == 0).mean() >= 0.999


@pytest.mark.parametrize("M,K,I", [(1, 5120, 17408), (2, 5120, 17408), (3, 512, 1024),
                                   (1, 256, 512)])
def test_rmsnorm_gate_up_swiglu(a8w8, M, K, I):
    """a11-a12 as the step runs them: the post-attention RMSNorm and the row's
    quantisation in the projection kernel's prologue, Gate/Up and SwiGLU."""
    seed = 3 * M + K + I
    x = synth.bf16_normal(seed, (M, K), std=40.0)
    nw = synth.bf16_normal(seed + 1, (K,), mean=1.0, std=0.02)
    W = synth.int8_uniform(seed + 2, (2 * I, K))
    s = synth.scales_uniform(seed + 3, 2 * I)
    act = to_host(a8w8.a8w8_rmsnorm_gate_up_swiglu(to_dev(x), to_dev(nw), 1e-6, to_dev(W),
                                                   to_dev(s)))
    xn = oracle.rmsnorm(x, nw, 1e-6)
    q, qs = oracle.quant_rows(xn)
    oact, _ = oracle.gate_up_swiglu(q, qs, W, s)
    # two-float norm and SiLU: one BF16 unit at most, 99.9% identical
    assert bf16_close(act, oact, 1, 1e-3).all()
    assert (bf16_ulp_diff(act, oact) == 0).mean() >= 0.999


# ---------------------------------------------------------------------------
# Exact INT32 product of prefill rows on the tensor cores (tcgen05)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,K,N,k0,k1", [
    (130, 320, 300, 0, 320),          # ragged M and N tiles, one partial chunk
    (200, 2112, 136, 0, 2112),        # 33 K steps: chunks of 16, 16 and 1 steps
    (64, 1024, 128, 0, 1024),         # exactly one chunk, one tile
    (257, 17408, 260, 8704, 17408),   # the down projection's second K half
    (2048, 5120, 256, 0, 5120),       # the prefill chunk's rows, Qwen3-14B K
])
def test_matmul_i8_exact(a8w8, M, K, N, k0, k1):
    x = synth.int8_uniform(M + K, (M, K))
    W = synth.int8_uniform(N + K + 1, (N, K))
    acc = to_host(a8w8.a8w8_matmul_i8(to_dev(x), to_dev(W), k0, k1))
    assert np.array_equal(acc, oracle.matmul_i8(x, W, k0, k1))
    assert a8w8.read_device_errors() == 0


@pytest.mark.parametrize("a,b", [(127, 127), (-128, -128), (127, -127), (-128, 127)])
def test_matmul_i8_extreme_chunks(a8w8, a, b):
    # every product at the extreme: each 1024-column chunk sums to +-2^24 or
    # just below, the largest FP32 partial the exact accumulation meets
    M, K, N = 130, 5120, 136
    x = np.full((M, K), a, np.int8)
    W = np.full((N, K), b, np.int8)
    x[3, ::7] = -a if a != -128 else 127
    acc = to_host(a8w8.a8w8_matmul_i8(to_dev(x), to_dev(W)))
    assert np.array_equal(acc, oracle.matmul_i8(x, W))


# ---------------------------------------------------------------------------
# KV write and attention
# ---------------------------------------------------------------------------

def test_paged_kv_write_exact(a8w8):
    Hkv, D, page, nblk = 8, 128, 128, 5
    T = 6
    k = synth.bf16_normal(1, (T, Hkv, D))
    v = synth.bf16_normal(2, (T, Hkv, D))
    slots = np.array([3, -1, 130, 639, 0, -1], np.int32)
    kc = synth.bf16_normal(3, (nblk * page, Hkv, D))
    vc = synth.bf16_normal(4, (nblk * page, Hkv, D))
    gk, gv = to_dev(kc), to_dev(vc)
    a8w8.paged_kv_write(to_dev(k), to_dev(v), to_dev(slots), gk, gv, page)
    okc, ovc = kc.copy(), vc.copy()
    assert oracle.kv_write(k, v, slots, okc, ovc) == 0
    assert np.array_equal(to_host(gk), okc) and np.array_equal(to_host(gv), ovc)
    assert a8w8.read_device_errors() == 0


def test_paged_kv_write_out_of_range_slot_is_flagged(a8w8):
    Hkv, D, page, nblk = 2, 64, 16, 2
    k = synth.bf16_normal(5, (2, Hkv, D))
    kc = np.zeros((nblk * page, Hkv, D), np.uint16)
    gk, gv = to_dev(kc), to_dev(kc)
    a8w8.read_device_errors()
    a8w8.paged_kv_write(to_dev(k), to_dev(k), to_dev(np.array([5, 32], np.int32)), gk, gv, page)
    assert a8w8.read_device_errors() & a8w8.DEVERR_SLOT
    out = to_host(gk)
    assert np.array_equal(out[5], k[0]) and not np.delete(out, 5, axis=0).any()


def _attn_case(seed, B, Hq, Hkv, D, page, ctx, spare=2):
    ctx = np.asarray(ctx, np.int32)
    bt, nblk = synth.paged_layout(seed, np.maximum(ctx, 1), page, spare_blocks=spare)
    kc = synth.kv_cache(seed + 1, nblk, page, Hkv, D)
    vc = synth.kv_cache(seed + 2, nblk, page, Hkv, D)
    q = synth.bf16_normal(seed + 3, (B, Hq, D))
    return q, kc, vc, bt, ctx


ATTN_CASES = [
    # B, Hq, Hkv, D, page, ctx
    (1, 40, 8, 128, 128, [256]),                  # one layer at max_seq_len 256
    (1, 40, 8, 128, 128, [1]),                    # single token: output = V
    (1, 4, 2, 64, 16, [16]),                      # tiny layer
    (4, 40, 8, 128, 128, [64, 4096, 1000, 129]),  # split-KV with a combine pass
    (3, 8, 8, 64, 16, [300, 0, 17]),              # MHA grouping, a padded row, splits
    (16, 40, 8, 128, 128, list(synth.batched_ctx_lens(5, 16))),
]


@pytest.mark.parametrize("B,Hq,Hkv,D,page,ctx", ATTN_CASES)
def test_paged_attention_vs_oracle(a8w8, B, Hq, Hkv, D, page, ctx):
    q, kc, vc, bt, ctxa = _attn_case(B * 31 + D, B, Hq, Hkv, D, page, ctx)
    out = a8w8.paged_decode_attention_bf16(to_dev(q), to_dev(kc), to_dev(vc), to_dev(bt),
                                           to_dev(ctxa), page)
    ref, rc = oracle.paged_attention(q, kc, vc, bt, ctxa, page)
    assert rc == 0
    g = to_host(out)
    for b in range(B):
        if ctxa[b] == 0:
            assert not g[b].any()
    # two-float softmax against the double oracle: one BF16 unit (of the
    # output's scale near zero) at most, 99.9% identical
    assert rel_l2(bf16_to_f64(g), bf16_to_f64(ref)) <= 2e-3
    assert bf16_close(g, ref, 1, 0.1).all()
    eq = (bf16_ulp_diff(g, ref) == 0).mean()
    print("identical fraction", eq)
    assert eq >= 0.999
    assert a8w8.read_device_errors() == 0


def test_paged_attention_shuffle_invariant(a8w8):
    B, Hq, Hkv, D, page = 2, 16, 2, 128, 128
    ctx = np.array([700, 301], np.int32)
    q, kc, vc, bt, _ = _attn_case(11, B, Hq, Hkv, D, page, ctx, spare=0)
    # the same logical cache laid out through a different permutation
    perm = np.random.default_rng(12).permutation(int(bt.max()) + 1).astype(np.int32)
    bt2 = perm[bt]
    kc2 = np.zeros_like(kc)
    vc2 = np.zeros_like(vc)
    for old, new in enumerate(perm):
        kc2[new * page:(new + 1) * page] = kc[old * page:(old + 1) * page]
        vc2[new * page:(new + 1) * page] = vc[old * page:(old + 1) * page]
    o1 = to_host(a8w8.paged_decode_attention_bf16(to_dev(q), to_dev(kc), to_dev(vc), to_dev(bt),
                                                  to_dev(ctx), page))
    o2 = to_host(a8w8.paged_decode_attention_bf16(to_dev(q), to_dev(kc2), to_dev(vc2),
                                                  to_dev(bt2), to_dev(ctx), page))
    assert np.array_equal(o1, o2)


def test_paged_attention_bad_block_is_flagged(a8w8):
    B, Hq, Hkv, D, page = 1, 4, 2, 64, 16
    q, kc, vc, bt, ctx = _attn_case(21, B, Hq, Hkv, D, page, [20])
    bt = bt.copy()
    bt[0, 1] = 10_000
    a8w8.read_device_errors()
    a8w8.paged_decode_attention_bf16(to_dev(q), to_dev(kc), to_dev(vc), to_dev(bt), to_dev(ctx), page)
    assert a8w8.read_device_errors() & a8w8.DEVERR_BLOCK


def test_rope_table(a8w8):
    for D in (64, 128):
        t = to_host(a8w8.a8w8_rope_table(4200, D, 1e6))
        pos = np.arange(4200, dtype=np.float64)[:, None]
        inv = 1e6 ** (-2.0 * np.arange(D // 2) / D)
        ang = pos * inv[None, :]
        c = t[:, : D // 2].astype(np.float64) + t[:, D: 3 * D // 2]
        s = t[:, D // 2: D].astype(np.float64) + t[:, 3 * D // 2:]
        np.testing.assert_allclose(t[:, : D // 2], np.cos(ang), atol=1e-7, rtol=0)
        np.testing.assert_allclose(t[:, D // 2: D], np.sin(ang), atol=1e-7, rtol=0)
        # hi + lo carries the device's double value to about 2^-48; that value
        # differs from numpy's by the few-ulp differences of pow/cos/sin at
        # angles up to ~4200 rad (~4200 * 2^-52 absolute)
        np.testing.assert_allclose(c, np.cos(ang), atol=1e-12, rtol=0)
        np.testing.assert_allclose(s, np.sin(ang), atol=1e-12, rtol=0)
        assert t.shape == (4200, 2 * D)
