"""The Python binding marshals every entry point with the arity and argument
types its ctypes signature declares.

No GPU is involved: the library is replaced by a recorder that checks each
call against the signature table (which test_abi.py ties to the header), and
CPU tensors stand in for device ones. This catches a wrapper that drops,
duplicates or reorders an argument before any kernel runs.
"""
import ctypes

import pytest

import synth
import w8a8_quantized_decode_gb300 as a8w8

torch = pytest.importorskip("torch")


class _Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        res, argtypes = a8w8._SIGNATURES[name]

        def f(*args):
            assert len(args) == len(argtypes), (name, len(args), len(argtypes))
            for i, (a, t) in enumerate(zip(args, argtypes)):
                if t in (ctypes.c_int, ctypes.c_size_t, ctypes.c_uint64):
                    assert isinstance(a, int) and not isinstance(a, bool), (name, i, a)
                elif t in (ctypes.c_float, ctypes.c_double):
                    assert isinstance(a, (int, float)), (name, i, a)
                elif t is ctypes.c_void_p:
                    assert (a is None or isinstance(a, (int, ctypes.Array))
                            or type(a).__name__ == "CArgObject"), (name, i, type(a))
            self.calls.append(name)
            return 0
        return f


@pytest.fixture
def rec(monkeypatch):
    r = _Recorder()
    monkeypatch.setattr(a8w8, "lib", lambda: r)
    monkeypatch.setattr(a8w8, "_ptr", lambda t: None if t is None else t.data_ptr())
    monkeypatch.setattr(a8w8, "_stream", lambda s=None: None)
    return r


CFG = dict(synth.TINY, num_layers=2, vocab=64)


def _t(shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def _caches(n=4):
    page, Hkv, D = CFG["page_size"], CFG["num_kv_heads"], CFG["head_dim"]
    return _t((n * page, Hkv, D))


def _i8_cache(n=4):
    page, Hkv, D = CFG["page_size"], CFG["num_kv_heads"], CFG["head_dim"]
    return _t((n * page, Hkv, D), torch.int8), _t((n * page, Hkv), torch.float32)


def _weights():
    return {k: torch.from_numpy(v.view("int16") if v.dtype.name == "uint16" else v)
            for k, v in synth.layer_weights(CFG, 1).items()}


def _bf16_weights():
    return {k: torch.from_numpy(v.view("int16")) for k, v in synth.bf16_layer_weights(CFG, 1).items()}


def _rows(B):
    i32 = torch.int32
    return _t((B,), i32), _t((B,), i32), _t((B, 2), i32), _t((B,), i32)


def test_int8_kv_wrappers(rec):
    kc, ks = _i8_cache()
    vc, vs = _i8_cache()
    Hkv, D = CFG["num_kv_heads"], CFG["head_dim"]
    a8w8.paged_kv_write_i8(_t((3, Hkv, D)), _t((3, Hkv, D)), _t((3,), torch.int32), kc, vc, ks, vs,
                           CFG["page_size"])
    q = _t((2, CFG["num_q_heads"], D))
    a8w8.paged_decode_attention_i8kv(q, kc, vc, ks, vs, _t((2, 2), torch.int32),
                                     _t((2,), torch.int32), CFG["page_size"], ws=_t((16,), torch.uint8))
    tok, slot, bt, ctx = _rows(2)
    rope, ws = _t((32, 2 * D), torch.float32), _t((64,), torch.uint8)
    hidden = _t((2, CFG["hidden"]))
    a8w8.a8w8_decode_layer_i8kv(_weights(), CFG, hidden, slot, bt, ctx, kc, vc, ks, vs, rope, ws,
                                taps={"xn": _t((2, CFG["hidden"]))})
    a8w8.a8w8_prefill_layer_i8kv(_weights(), CFG, hidden, slot, bt, ctx, kc, vc, ks, vs, rope, ws)
    model = {"embed": _t((64, CFG["hidden"])), "final_norm_w": _t((CFG["hidden"],)),
             "lm_head": _t((64, CFG["hidden"])), "layers": [_weights(), _weights()]}
    a8w8.a8w8_decode_step_i8kv(model, CFG, tok, slot, bt, ctx, [kc, kc], [vc, vc], [ks, ks],
                               [vs, vs], rope, ws, _t((2,), torch.int32))
    assert rec.calls == ["paged_kv_write_i8", "a8w8_attention_workspace_bytes",
                         "paged_decode_attention_i8kv",
                         "a8w8_decode_layer_i8kv", "a8w8_prefill_layer_i8kv",
                         "a8w8_decode_step_i8kv"]


def test_bf16_layer_and_prefill_step_wrappers(rec):
    H, I, D = CFG["hidden"], CFG["intermediate"], CFG["head_dim"]
    x = _t((3, H))
    a8w8.bf16_linear(x, _t((5, H)), residual=_t((3, 5)))
    a8w8.bf16_gate_up_swiglu(x, _t((2 * I, H)))
    tok, slot, bt, ctx = _rows(2)
    rope, ws = _t((32, 2 * D), torch.float32), _t((64,), torch.uint8)
    a8w8.bf16_decode_layer(_bf16_weights(), CFG, _t((2, H)), slot, bt, ctx, _caches(), _caches(),
                           rope, ws)
    model = {"embed": _t((64, H)), "final_norm_w": _t((H,)), "lm_head": _t((64, H)),
             "layers": [_weights(), _weights()]}
    a8w8.a8w8_prefill_step(model, CFG, tok, slot, bt, ctx, [_caches()] * 2, [_caches()] * 2, rope,
                           ws, _t((1,), torch.int32), _t((1,), torch.int32))
    assert rec.calls == ["bf16_linear", "bf16_gate_up_swiglu", "bf16_decode_layer",
                         "a8w8_prefill_step"]


def test_measured_path_wrappers(rec):
    D, H, I = CFG["head_dim"], CFG["hidden"], CFG["intermediate"]
    a8w8.a8w8_rmsnorm_gate_up_swiglu(_t((2, H)), _t((H,)), 1e-6, _t((2 * I, H), torch.int8),
                                     _t((2 * I,), torch.float32))
    a8w8.a8w8_matmul_i8(_t((3, H), torch.int8), _t((5, H), torch.int8), 0, H)
    tok, slot, bt, ctx = _rows(2)
    rope, ws = _t((32, 2 * D), torch.float32), _t((64,), torch.uint8)
    a8w8.a8w8_decode_layer(_weights(), CFG, _t((2, CFG["hidden"])), slot, bt, ctx, _caches(),
                           _caches(), rope, ws)
    a8w8.a8w8_prefill_layer(_weights(), CFG, _t((2, CFG["hidden"])), slot, bt, ctx, _caches(),
                            _caches(), rope, ws)
    model = {"embed": _t((64, CFG["hidden"])), "final_norm_w": _t((CFG["hidden"],)),
             "lm_head": _t((64, CFG["hidden"])), "layers": [_weights(), _weights()]}
    a8w8.a8w8_decode_step(model, CFG, tok, slot, bt, ctx, [_caches()] * 2, [_caches()] * 2, rope,
                          ws, _t((2,), torch.int32))
    assert rec.calls == ["a8w8_rmsnorm_gate_up_swiglu", "a8w8_matmul_i8", "a8w8_decode_layer",
                         "a8w8_prefill_layer", "a8w8_decode_step"]
