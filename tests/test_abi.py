"""The C-ABI library loads, exports every declared entry point, and rejects bad
arguments on the host before touching the GPU (no compute call is made)."""
import ctypes

import pytest

import synth
import w8a8_quantized_decode_gb300 as a8w8


@pytest.fixture(scope="module")
def lib():
    a8w8.build()
    return a8w8.lib()


def test_every_declared_symbol_is_exported(lib):
    names = a8w8.header_functions()
    assert len(names) >= 17
    for n in names:
        assert hasattr(lib, n), n
    # the binding wraps every declared entry point
    assert set(names) <= set(a8w8._SIGNATURES)


def test_version(lib):
    assert lib.a8w8_version() == 100


FAKE = 0x10000   # a 16-byte aligned non-null address; never dereferenced by the host checks


def test_linear_validation(lib):
    L = lib
    assert L.a8w8_linear(None, FAKE, 1, 32, FAKE, FAKE, 4, 1, None, FAKE, None, None) == a8w8.ERR_INVALID_ARG
    assert b"NULL" in L.a8w8_last_error()
    assert L.a8w8_linear(FAKE, FAKE, 1, 24, FAKE, FAKE, 4, 1, None, FAKE, None, None) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert L.a8w8_linear(FAKE, FAKE, 1, 32, FAKE, FAKE, 4, 3, None, FAKE, None, None) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert L.a8w8_linear(FAKE, FAKE, 1, 48, FAKE, FAKE, 4, 2, None, FAKE, None, None) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert L.a8w8_linear(FAKE + 4, FAKE, 1, 32, FAKE, FAKE, 4, 1, None, FAKE, None, None) == a8w8.ERR_INVALID_ARG
    assert L.a8w8_linear(FAKE, FAKE, -1, 32, FAKE, FAKE, 4, 1, None, FAKE, None, None) == a8w8.ERR_INVALID_ARG
    # empty problems are a no-op
    assert L.a8w8_linear(None, None, 0, 32, None, None, 4, 1, None, None, None, None) == a8w8.OK
    assert L.a8w8_gate_up_swiglu(FAKE, FAKE, 1, 20, FAKE, FAKE, 4, FAKE, None, None) == a8w8.ERR_UNSUPPORTED_SHAPE


def test_matmul_i8_validation(lib):
    f = lib.a8w8_matmul_i8
    assert f(FAKE, 4, 96, FAKE, 4, 0, 96, FAKE, FAKE, None) == a8w8.ERR_UNSUPPORTED_SHAPE   # K % 64
    assert f(FAKE, 4, 128, FAKE, 4, 32, 128, FAKE, FAKE, None) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert f(FAKE, 4, 128, FAKE, 4, 0, 192, FAKE, FAKE, None) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert f(FAKE, 4, 128, FAKE, 4, 64, 64, FAKE, FAKE, None) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert f(FAKE + 8, 4, 128, FAKE, 4, 0, 128, FAKE, FAKE, None) == a8w8.ERR_INVALID_ARG
    assert f(FAKE, 4, 128, None, 4, 0, 128, FAKE, FAKE, None) == a8w8.ERR_INVALID_ARG
    assert f(FAKE, -1, 128, FAKE, 4, 0, 128, FAKE, FAKE, None) == a8w8.ERR_INVALID_ARG
    assert f(FAKE, 4, 128, FAKE, 4, 0, 128, FAKE, None, None) == a8w8.ERR_INVALID_ARG   # scratch
    assert f(None, 0, 128, None, 4, 0, 128, None, None, None) == a8w8.OK


def test_rmsnorm_gate_up_validation(lib):
    L = lib
    f = L.a8w8_rmsnorm_gate_up_swiglu
    assert f(FAKE, 1, 20, FAKE, 1e-6, FAKE, FAKE, 4, FAKE, None) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert f(FAKE, 1, 65552, FAKE, 1e-6, FAKE, FAKE, 4, FAKE, None) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert f(FAKE, 1, 32, None, 1e-6, FAKE, FAKE, 4, FAKE, None) == a8w8.ERR_INVALID_ARG
    assert f(FAKE, 1, 32, FAKE, -1.0, FAKE, FAKE, 4, FAKE, None) == a8w8.ERR_INVALID_ARG
    assert f(FAKE, -1, 32, FAKE, 1e-6, FAKE, FAKE, 4, FAKE, None) == a8w8.ERR_INVALID_ARG
    assert f(None, 0, 32, None, 1e-6, None, None, 4, None, None) == a8w8.OK


def test_quant_and_kv_validation(lib):
    L = lib
    assert L.a8w8_quant_rows(FAKE, 2, 12, 12, FAKE, FAKE, None) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert L.a8w8_quant_rows(FAKE, 2, 16, 8, FAKE, FAKE, None) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert L.a8w8_quant_rows(None, 2, 16, 16, FAKE, FAKE, None) == a8w8.ERR_INVALID_ARG
    assert L.a8w8_quant_rows(None, 0, 16, 16, None, None, None) == a8w8.OK
    assert L.paged_kv_write(FAKE, FAKE, 1, 1, 4, FAKE, FAKE, FAKE, 1, 16, None) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert L.paged_kv_write(None, FAKE, 1, 2, 64, FAKE, FAKE, FAKE, 1, 16, None) == a8w8.ERR_INVALID_ARG
    assert L.paged_kv_write(None, None, 0, 2, 64, None, None, None, 1, 16, None) == a8w8.OK


def test_attention_validation(lib):
    L = lib
    args = lambda D, Hq, Hkv, ws, wsb: (FAKE, FAKE, FAKE, FAKE, FAKE, 2, Hq, Hkv, D, 128, 40, 100,
                                        0.1, FAKE, ws, wsb, None)
    assert L.paged_decode_attention_bf16(*args(96, 8, 2, None, 0)) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert L.paged_decode_attention_bf16(*args(128, 9, 2, None, 0)) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert L.paged_decode_attention_bf16(*args(128, 32, 2, None, 0)) == a8w8.ERR_UNSUPPORTED_SHAPE
    # 40 blocks of 128 tokens need split-KV partials: a missing workspace is reported
    need = L.a8w8_attention_workspace_bytes(2, 8, 128, 40 * 128)
    assert need > 0
    assert L.paged_decode_attention_bf16(*args(128, 8, 2, None, 0)) == a8w8.ERR_WORKSPACE
    assert L.paged_decode_attention_bf16(*args(128, 8, 2, FAKE, need - 1)) == a8w8.ERR_WORKSPACE
    # short contexts need none
    assert L.a8w8_attention_workspace_bytes(1, 40, 128, 256) == 0


def _cfg(c):
    return ctypes.byref(a8w8.make_config(c))


def test_workspace_sizes(lib):
    q = synth.QWEN3_14B
    small = lib.a8w8_workspace_bytes(_cfg(q), 1, 2)
    big = lib.a8w8_workspace_bytes(_cfg(q), 16, 33)
    assert 0 < small < big
    # at least the activations the layer keeps: qkv, attention output, SwiGLU output, hidden
    H, I = q["hidden"], q["intermediate"]
    assert small >= 2 * (H + 7168 + 40 * 128 + I)
    assert lib.a8w8_workspace_bytes(None, 1, 1) == 0
    assert lib.a8w8_workspace_bytes(_cfg(q), 0, 1) == 0


def test_layer_and_step_validation(lib):
    L = lib
    q = synth.QWEN3_14B
    w = a8w8.LayerWeights(*([FAKE] * len(a8w8.WEIGHT_FIELDS)))
    base = dict(B=1, max_blocks=2, num_blocks=4, rope=FAKE, max_pos=256, ws=FAKE, wsb=1 << 30)

    def call(cfg, w=w, **kw):
        a = dict(base, **kw)
        return L.a8w8_decode_layer(ctypes.byref(w), _cfg(cfg), a["B"], FAKE, FAKE, FAKE,
                                   a["max_blocks"], a["num_blocks"], FAKE, FAKE, FAKE, a["rope"],
                                   a["max_pos"], a["ws"], a["wsb"], None, None)
    assert call(dict(q, head_dim=96)) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert call(dict(q, num_kv_heads=7)) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert call(dict(q, down_k_splits=3)) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert call(dict(q, hidden=5128)) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert call(q, B=0) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert call(q, B=65) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert call(q, rope=None) == a8w8.ERR_INVALID_ARG
    assert call(q, wsb=1000) == a8w8.ERR_WORKSPACE
    bad = a8w8.LayerWeights(*([FAKE] * len(a8w8.WEIGHT_FIELDS)))
    bad.w_down = None
    assert call(q, w=bad) == a8w8.ERR_INVALID_ARG
    assert L.a8w8_decode_layer(None, _cfg(q), 1, FAKE, FAKE, FAKE, 2, 4, FAKE, FAKE, FAKE, FAKE,
                               256, FAKE, 1 << 30, None, None) == a8w8.ERR_INVALID_ARG

    # step: null model, and vocab must be set
    caches = (ctypes.c_void_p * 1)(FAKE)
    assert L.a8w8_decode_step(None, _cfg(dict(q, num_layers=1)), 1, FAKE, FAKE, FAKE, 2, 4, FAKE,
                              caches, caches, FAKE, 256, FAKE, None, None, FAKE, 1 << 30,
                              None) == a8w8.ERR_INVALID_ARG
    layers = (a8w8.LayerWeights * 1)(w)
    m = a8w8.Model(FAKE, ctypes.cast(layers, ctypes.c_void_p), FAKE, FAKE)
    assert L.a8w8_decode_step(ctypes.byref(m), _cfg(dict(q, num_layers=1, vocab=0)), 1, FAKE, FAKE,
                              FAKE, 2, 4, FAKE, caches, caches, FAKE, 256, FAKE, None, None, FAKE,
                              1 << 30, None) == a8w8.ERR_INVALID_ARG
    assert L.a8w8_decode_step(ctypes.byref(m), _cfg(dict(q, num_layers=1)), 1, FAKE, FAKE, FAKE, 2,
                              4, FAKE, caches, caches, FAKE, 256, FAKE, None, None, FAKE, 100,
                              None) == a8w8.ERR_WORKSPACE
    # graph creation validates the same way and returns no handle
    out = ctypes.c_void_p(123)
    assert L.a8w8_step_graph_create(ctypes.byref(out), ctypes.byref(m),
                                    _cfg(dict(q, num_layers=1)), 1, 2, 4, caches, caches, FAKE,
                                    256, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 1, FAKE, 100,
                                    None) == a8w8.ERR_WORKSPACE
    assert out.value is None
    assert L.a8w8_step_graph_launch(None, None) == a8w8.ERR_INVALID_ARG
    L.a8w8_step_graph_destroy(None)

    # sampled graph: its own arguments are checked before anything is captured
    def sampled(**kw):
        a = dict(logits=FAKE, T=1.0, top_p=0.9, ctr=FAKE, sws=FAKE, swsb=1 << 30, wsb=1 << 30)
        a.update(kw)
        o = ctypes.c_void_p(123)
        r = L.a8w8_step_graph_create_sampled(
            ctypes.byref(o), ctypes.byref(m), _cfg(dict(q, num_layers=1)), 1, 2, 4, caches, caches,
            FAKE, 256, FAKE, FAKE, FAKE, FAKE, FAKE, a["logits"], None, 1, a["T"], a["top_p"], 7,
            a["ctr"], a["sws"], a["swsb"], FAKE, a["wsb"], None)
        assert o.value is None
        return r
    assert sampled(logits=None) == a8w8.ERR_INVALID_ARG
    assert sampled(ctr=None) == a8w8.ERR_INVALID_ARG
    assert sampled(ctr=FAKE + 4) == a8w8.ERR_INVALID_ARG
    assert sampled(T=float("nan")) == a8w8.ERR_INVALID_ARG
    assert sampled(top_p=0.0) == a8w8.ERR_INVALID_ARG
    assert sampled(top_p=1.5) == a8w8.ERR_INVALID_ARG
    assert sampled(sws=None) == a8w8.ERR_WORKSPACE
    assert sampled(swsb=100) == a8w8.ERR_WORKSPACE
    assert sampled(wsb=100) == a8w8.ERR_WORKSPACE   # then the step's own checks


def test_rope_table_validation(lib):
    assert lib.a8w8_rope_table(FAKE, 16, 63, 1e6, None) == a8w8.ERR_INVALID_ARG
    assert lib.a8w8_rope_table(FAKE, 16, 64, 0.0, None) == a8w8.ERR_INVALID_ARG
    assert lib.a8w8_rope_table(None, 16, 64, 1e6, None) == a8w8.ERR_INVALID_ARG
    assert lib.a8w8_rope_table(None, 0, 64, 1e6, None) == a8w8.OK


def test_prefill_layer_validation(lib):
    L = lib
    q = synth.QWEN3_14B
    w = a8w8.LayerWeights(*([FAKE] * len(a8w8.WEIGHT_FIELDS)))

    def call(cfg, M=64, max_blocks=4, wsb=1 << 34, wptr=w):
        return L.a8w8_prefill_layer(ctypes.byref(wptr), _cfg(cfg), M, FAKE, FAKE, FAKE, max_blocks,
                                    8, FAKE, FAKE, FAKE, FAKE, 512, FAKE, wsb, None, None)
    assert call(q, M=0) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert call(q, M=16385) == a8w8.ERR_UNSUPPORTED_SHAPE
    # grouped attention: at most 7 query heads per KV head, 64 chunks of 128 tokens
    assert call(dict(q, num_kv_heads=5)) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert call(q, max_blocks=65) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert b"prefill attention" in L.a8w8_last_error()
    # the workspace grows with M (the GEMM's INT32 results for M > 64 rows)
    need = L.a8w8_workspace_bytes(_cfg(q), 2048, 4)
    assert need > L.a8w8_workspace_bytes(_cfg(q), 64, 4) * 8
    assert call(q, M=2048, wsb=need - 1) == a8w8.ERR_WORKSPACE
    nullw = a8w8.LayerWeights(*([None] * len(a8w8.WEIGHT_FIELDS)))
    assert call(q, wptr=nullw) == a8w8.ERR_INVALID_ARG


def test_sample_validation(lib):
    L = lib
    ok = dict(B=2, V=10, ld=10, T=1.0, p=0.9, ws=FAKE, wsb=1 << 20)

    def call(**kw):
        a = dict(ok, **kw)
        return L.a8w8_sample(FAKE, a["B"], a["V"], a["ld"], a["T"], a["p"], 1, 2, FAKE, a["ws"],
                             a["wsb"], None)
    assert call(p=0.0) == a8w8.ERR_INVALID_ARG
    assert call(p=1.5) == a8w8.ERR_INVALID_ARG
    assert call(T=float("nan")) == a8w8.ERR_INVALID_ARG
    assert call(ld=5) == a8w8.ERR_INVALID_ARG
    assert call(B=0) == a8w8.OK
    assert call(ws=None, wsb=0) == a8w8.ERR_WORKSPACE
    assert call(T=0.0, ws=None, wsb=0) == a8w8.ERR_WORKSPACE
    need = L.a8w8_sample_workspace_bytes(2, 10)
    assert need >= 2 * 10 * 8 and L.a8w8_sample_workspace_bytes(2, 20) - need == 2 * 10 * 8
    assert call(wsb=need - 1) == a8w8.ERR_WORKSPACE


def test_int8_kv_validation(lib):
    L = lib
    # quantise-on-write: head_dim 64 or 128, every pointer given and aligned
    args = lambda D, k=FAKE, ks=FAKE: (k, FAKE, 2, 8, D, FAKE, FAKE, FAKE, ks, FAKE, 4, 16, None)
    assert L.paged_kv_write_i8(*args(96)) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert L.paged_kv_write_i8(*args(128, k=None)) == a8w8.ERR_INVALID_ARG
    assert L.paged_kv_write_i8(*args(128, ks=FAKE + 4)) == a8w8.ERR_INVALID_ARG
    assert L.paged_kv_write_i8(None, None, 0, 8, 128, None, None, None, None, None, 4, 16,
                               None) == a8w8.OK
    # attention: the BF16 form's shape and workspace rules
    att = lambda D, Hq, ws, wsb, vs=FAKE: (FAKE, FAKE, FAKE, FAKE, vs, FAKE, FAKE, 2, Hq, 2, D,
                                           128, 40, 100, 0.1, FAKE, ws, wsb, None)
    assert L.paged_decode_attention_i8kv(*att(96, 8, None, 0)) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert L.paged_decode_attention_i8kv(*att(128, 32, None, 0)) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert L.paged_decode_attention_i8kv(*att(128, 8, FAKE, 1 << 30, vs=None)) == a8w8.ERR_INVALID_ARG
    need = L.a8w8_attention_workspace_bytes(2, 8, 128, 40 * 128)
    assert L.paged_decode_attention_i8kv(*att(128, 8, FAKE, need - 1)) == a8w8.ERR_WORKSPACE
    # layer: the decode layer's checks, plus the four cache pointers
    q = synth.QWEN3_14B
    w = a8w8.LayerWeights(*([FAKE] * len(a8w8.WEIGHT_FIELDS)))

    def layer(cfg, B=1, kc=FAKE, wsb=1 << 30):
        return L.a8w8_decode_layer_i8kv(ctypes.byref(w), _cfg(cfg), B, FAKE, FAKE, FAKE, 2, 4, FAKE,
                                        kc, FAKE, FAKE, FAKE, FAKE, 256, FAKE, wsb, None, None)
    assert layer(dict(q, head_dim=96)) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert layer(q, B=65) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert layer(q, kc=None) == a8w8.ERR_INVALID_ARG
    assert layer(q, wsb=1000) == a8w8.ERR_WORKSPACE


def test_bf16_layer_validation(lib):
    L = lib
    assert L.bf16_linear(FAKE, 1, 20, FAKE, 4, None, FAKE, None) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert L.bf16_linear(FAKE, 1, 49160, FAKE, 4, None, FAKE, None) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert L.bf16_linear(None, 1, 32, FAKE, 4, None, FAKE, None) == a8w8.ERR_INVALID_ARG
    assert L.bf16_linear(FAKE, 1, 32, FAKE, 4, FAKE + 2, FAKE, None) == a8w8.ERR_INVALID_ARG
    assert L.bf16_linear(None, 0, 32, None, 4, None, None, None) == a8w8.OK
    assert L.bf16_gate_up_swiglu(FAKE, 1, 12, FAKE, 4, FAKE, None) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert L.bf16_gate_up_swiglu(FAKE, 1, 32, None, 4, FAKE, None) == a8w8.ERR_INVALID_ARG
    q = synth.QWEN3_14B
    w = a8w8.Bf16LayerWeights(*([FAKE] * len(a8w8.BF16_WEIGHT_FIELDS)))

    def layer(cfg, w=w, B=1, wsb=1 << 30):
        return L.bf16_decode_layer(ctypes.byref(w), _cfg(cfg), B, FAKE, FAKE, FAKE, 2, 4, FAKE, FAKE,
                                   FAKE, FAKE, 256, FAKE, wsb, None, None)
    assert layer(dict(q, head_dim=96)) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert layer(q, B=65) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert layer(dict(q, intermediate=49168)) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert layer(q, wsb=1000) == a8w8.ERR_WORKSPACE
    bad = a8w8.Bf16LayerWeights(*([FAKE] * len(a8w8.BF16_WEIGHT_FIELDS)))
    bad.w_down = None
    assert layer(q, w=bad) == a8w8.ERR_INVALID_ARG


def test_int8_kv_prefill_validation(lib):
    L = lib
    q = synth.QWEN3_14B
    w = a8w8.LayerWeights(*([FAKE] * len(a8w8.WEIGHT_FIELDS)))

    def call(cfg, M=64, max_blocks=4, ks=FAKE, wsb=1 << 34):
        return L.a8w8_prefill_layer_i8kv(ctypes.byref(w), _cfg(cfg), M, FAKE, FAKE, FAKE,
                                         max_blocks, 8, FAKE, FAKE, FAKE, ks, FAKE, FAKE, 512,
                                         FAKE, wsb, None, None)
    assert call(q, M=0) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert call(dict(q, num_kv_heads=5)) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert call(q, max_blocks=65) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert call(q, ks=None) == a8w8.ERR_INVALID_ARG
    need = L.a8w8_workspace_bytes(_cfg(q), 2048, 4)
    assert call(q, M=2048, wsb=need - 1) == a8w8.ERR_WORKSPACE


def test_int8_kv_step_validation(lib):
    L = lib
    q = dict(synth.QWEN3_14B, num_layers=1)
    w = a8w8.LayerWeights(*([FAKE] * len(a8w8.WEIGHT_FIELDS)))
    layers = (a8w8.LayerWeights * 1)(w)
    m = a8w8.Model(FAKE, ctypes.cast(layers, ctypes.c_void_p), FAKE, FAKE)
    arr = (ctypes.c_void_p * 1)(FAKE)
    nul = (ctypes.c_void_p * 1)(None)

    def call(ks=arr, kc=arr, wsb=1 << 30):
        return L.a8w8_decode_step_i8kv(ctypes.byref(m), _cfg(q), 1, FAKE, FAKE, FAKE, 2, 4, FAKE,
                                       kc, arr, ks, arr, FAKE, 256, FAKE, None, None, FAKE, wsb,
                                       None)
    assert call(kc=nul) == a8w8.ERR_INVALID_ARG
    assert call(ks=nul) == a8w8.ERR_INVALID_ARG
    assert call(ks=None) == a8w8.ERR_INVALID_ARG
    assert call(wsb=100) == a8w8.ERR_WORKSPACE


def test_prefill_step_validation(lib):
    L = lib
    q = dict(synth.QWEN3_14B, num_layers=1)
    w = a8w8.LayerWeights(*([FAKE] * len(a8w8.WEIGHT_FIELDS)))
    layers = (a8w8.LayerWeights * 1)(w)
    m = a8w8.Model(FAKE, ctypes.cast(layers, ctypes.c_void_p), FAKE, FAKE)
    arr = (ctypes.c_void_p * 1)(FAKE)

    def call(cfg=q, M=512, S=1, max_blocks=8, last=FAKE, wsb=1 << 34):
        return L.a8w8_prefill_step(ctypes.byref(m), _cfg(cfg), M, FAKE, FAKE, FAKE, max_blocks, 16,
                                   FAKE, arr, arr, FAKE, 1024, S, last, FAKE, None, FAKE, wsb, None)
    assert call(M=0) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert call(S=0) == a8w8.ERR_INVALID_ARG
    assert call(S=513) == a8w8.ERR_INVALID_ARG
    assert call(max_blocks=65) == a8w8.ERR_UNSUPPORTED_SHAPE
    assert call(last=None) == a8w8.ERR_INVALID_ARG
    need = L.a8w8_workspace_bytes(_cfg(q), 512, 8)
    assert call(wsb=need - 1) == a8w8.ERR_WORKSPACE
