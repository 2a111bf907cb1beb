"""CPU oracle for the A8W8 decode layer and step (test infrastructure).

This package is the slow reference that the CUDA path is checked against. Only
the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it. It shares no code with the CUDA library: the C
source ``a8w8_oracle.c`` restates each step of the method (see the citations
there) and this module only marshals numpy arrays into it.

BF16 tensors are numpy ``uint16`` arrays holding the bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "a8w8_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liba8w8_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE float semantics, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            _declare(lib)
            _lib = lib
    return _lib


_p = ctypes.c_void_p
_i = ctypes.c_int
_l = ctypes.c_long
_d = ctypes.c_double


class Config(ctypes.Structure):
    _fields_ = [("hidden", _i), ("num_q_heads", _i), ("num_kv_heads", _i),
                ("head_dim", _i), ("intermediate", _i), ("num_layers", _i),
                ("vocab", _i), ("page_size", _i), ("down_k_splits", _i),
                ("rms_eps", _d), ("rope_theta", _d)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, _p) for n in (
        "input_norm_w", "w_qkv", "s_qkv", "q_norm_w", "k_norm_w", "w_o", "s_o",
        "post_norm_w", "w_gate_up", "s_gate_up", "w_down", "s_down")]


BF16_WEIGHT_NAMES = ("input_norm_w", "w_qkv", "q_norm_w", "k_norm_w", "w_o", "post_norm_w",
                     "w_gate_up", "w_down")


class LayerWeightsBF16(ctypes.Structure):
    _fields_ = [(n, _p) for n in BF16_WEIGHT_NAMES]


TAP_NAMES = ("xn", "xq", "xs", "acc_qkv", "qkv", "q_rot", "k_rot", "attn", "aq",
             "as", "acc_o", "h1", "hn", "hq", "hs", "acc_gu", "act", "actq",
             "acts", "acc_down")


class LayerTaps(ctypes.Structure):
    _fields_ = [(n, _p) for n in TAP_NAMES]


class Model(ctypes.Structure):
    _fields_ = [("embed", _p), ("layers", _p), ("final_norm_w", _p),
                ("lm_head", _p)]


def _declare(lib):
    sig = {
        "or_bf16_to_double": (_d, [ctypes.c_uint16]),
        "or_bf16_from_double": (ctypes.c_uint16, [_d]),
        "or_bf16_from_double_array": (None, [_p, _l, _p]),
        "or_rmsnorm": (None, [_p, _p, _i, _i, _d, _p]),
        "or_quant_rows": (None, [_p, _i, _i, _p, _p]),
        "or_matmul_i8": (_i, [_p, _i, _i, _p, _i, _i, _i, _p]),
        "or_dequant": (ctypes.c_float, [ctypes.c_int32, ctypes.c_float, ctypes.c_float]),
        "or_linear": (_i, [_p, _p, _i, _i, _p, _p, _i, _i, _p, _p, _p]),
        "or_gate_up_swiglu": (_i, [_p, _p, _i, _i, _p, _p, _i, _p, _p]),
        "or_rope": (None, [_p, _i, _i, _i, _p, _d]),
        "or_kv_write": (_i, [_p, _p, _i, _i, _i, _p, _p, _p, _l]),
        "or_paged_attention": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i,
                                    _d, _p]),
        "or_kv_write_i8": (_i, [_p, _p, _i, _i, _i, _p, _p, _p, _p, _p, _l]),
        "or_paged_attention_i8": (_i, [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i,
                                       _i, _i, _d, _p]),
        "or_decode_layer": (_i, [_p, _p, _i, _p, _p, _p, _i, _i, _p, _p, _p, _p]),
        "or_decode_layer_i8kv": (_i, [_p, _p, _i, _p, _p, _p, _i, _i, _p, _p, _p, _p, _p,
                                      _p]),
        "or_linear_bf16": (None, [_p, _i, _i, _p, _i, _p, _p]),
        "or_gate_up_swiglu_bf16": (None, [_p, _i, _i, _p, _i, _p]),
        "or_decode_layer_bf16": (_i, [_p, _p, _i, _p, _p, _p, _i, _i, _p, _p, _p, _p]),
        "or_argmax_f64": (None, [_p, _i, _i, _p]),
        "or_argmax_f32": (None, [_p, _i, _i, _p]),
        "or_lm_head": (None, [_p, _i, _i, _p, _i, _p]),
        "or_decode_step": (_i, [_p, _p, _i, _p, _p, _p, _i, _i, _p, _p, _p, _p, _p,
                                _p]),
        "or_num_threads": (_i, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    assert a.dtype == dtype, f"expected {dtype}, got {a.dtype}"
    return a


U16, I8, I32, F32 = np.uint16, np.int8, np.int32, np.float32


def num_threads() -> int:
    return _load().or_num_threads()


def bf16_from_f64(x) -> np.ndarray:
    """Round float64 values to BF16 bit patterns (RNE)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(x.shape, dtype=U16)
    _load().or_bf16_from_double_array(_ptr(x), x.size, _ptr(y))
    return y


def bf16_to_f64(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=U16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rmsnorm(x, w, eps: float) -> np.ndarray:
    x = _c(x, U16)
    w = _c(w, U16)
    cols = x.shape[-1]
    rows = x.size // cols
    assert w.size == cols
    y = np.empty_like(x)
    _load().or_rmsnorm(_ptr(x), _ptr(w), rows, cols, eps, _ptr(y))
    return y


def quant_rows(x):
    """Per-row dynamic INT8 quantisation of a BF16 matrix -> (q int8, scale f32)."""
    x = _c(x, U16)
    cols = x.shape[-1]
    rows = x.size // cols
    q = np.empty(x.shape, dtype=I8)
    s = np.empty(x.shape[:-1] if x.ndim > 1 else (1,), dtype=F32)
    _load().or_quant_rows(_ptr(x), rows, cols, _ptr(q), _ptr(s))
    return q, s


def matmul_i8(x, W, k_begin=0, k_end=None) -> np.ndarray:
    x = _c(x, I8)
    W = _c(W, I8)
    M, K = x.shape
    N = W.shape[0]
    assert W.shape[1] == K
    k_end = K if k_end is None else k_end
    acc = np.empty((M, N), dtype=I32)
    ov = _load().or_matmul_i8(_ptr(x), M, K, _ptr(W), N, k_begin, k_end, _ptr(acc))
    if ov:
        raise OverflowError("int32 accumulator overflow")
    return acc


def dequant(acc: int, s_act: float, s_w: float) -> np.float32:
    return np.float32(_load().or_dequant(int(acc), float(s_act), float(s_w)))


def linear(xq, xs, W, ws, k_splits: int = 1, residual=None):
    """A8W8 projection -> (y bf16 [M,N], full-K int32 acc [M,N])."""
    xq = _c(xq, I8)
    xs = _c(xs, F32)
    W = _c(W, I8)
    ws = _c(ws, F32)
    M, K = xq.shape
    N = W.shape[0]
    res = None if residual is None else _c(residual, U16)
    y = np.empty((M, N), dtype=U16)
    acc = np.empty((M, N), dtype=I32)
    rc = _load().or_linear(_ptr(xq), _ptr(xs), M, K, _ptr(W), _ptr(ws), N, k_splits,
                           _ptr(res), _ptr(y), _ptr(acc))
    if rc < 0:
        raise ValueError("K must be a multiple of k_splits")
    if rc > 0:
        raise OverflowError("int32 accumulator overflow")
    return y, acc


def gate_up_swiglu(xq, xs, W_gu, s_gu):
    xq = _c(xq, I8)
    xs = _c(xs, F32)
    W_gu = _c(W_gu, I8)
    s_gu = _c(s_gu, F32)
    M, K = xq.shape
    I = W_gu.shape[0] // 2
    act = np.empty((M, I), dtype=U16)
    acc = np.empty((M, 2 * I), dtype=I32)
    rc = _load().or_gate_up_swiglu(_ptr(xq), _ptr(xs), M, K, _ptr(W_gu), _ptr(s_gu), I,
                                   _ptr(act), _ptr(acc))
    if rc:
        raise OverflowError("int32 accumulator overflow")
    return act, acc


def rope(x, pos, theta: float):
    """RoPE on x [T, heads, D] (bf16) at per-token positions pos [T]; returns a copy."""
    y = _c(x, U16).copy()
    T, heads, D = y.shape
    pos = _c(pos, I32)
    _load().or_rope(_ptr(y), T, heads, D, _ptr(pos), theta)
    return y


def kv_write(k, v, slot_mapping, k_cache, v_cache) -> int:
    """Write k, v [T, Hkv, D] into the caches [slots, Hkv, D] in place."""
    k = _c(k, U16)
    v = _c(v, U16)
    sm = _c(slot_mapping, I32)
    assert k_cache.flags["C_CONTIGUOUS"] and v_cache.flags["C_CONTIGUOUS"]
    T, Hkv, D = k.shape
    num_slots = k_cache.size // (Hkv * D)
    return _load().or_kv_write(_ptr(k), _ptr(v), T, Hkv, D, _ptr(sm), _ptr(k_cache),
                               _ptr(v_cache), num_slots)


def paged_attention(q, k_cache, v_cache, block_table, ctx_lens, page: int,
                    scale: float | None = None):
    """q [B,Hq,D]; caches [num_blocks*page, Hkv, D]; returns (out [B,Hq,D], rc)."""
    q = _c(q, U16)
    k_cache = _c(k_cache, U16)
    v_cache = _c(v_cache, U16)
    bt = _c(block_table, I32)
    cl = _c(ctx_lens, I32)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[-2]
    num_blocks = k_cache.size // (Hkv * D * page)
    max_blocks = bt.shape[1]
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    out = np.empty_like(q)
    rc = _load().or_paged_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt),
                                    _ptr(cl), B, Hq, Hkv, D, page, max_blocks,
                                    num_blocks, scale, _ptr(out))
    return out, rc


def kv_write_i8(k, v, slot_mapping, k_codes, v_codes, k_scale, v_scale) -> int:
    """INT8 KV variant: quantise each K/V head row of k, v [T, Hkv, D] into
    codes [slots, Hkv, D] (int8) and row scales [slots, Hkv] (float32), in place."""
    k = _c(k, U16)
    v = _c(v, U16)
    sm = _c(slot_mapping, I32)
    for a, dt in ((k_codes, I8), (v_codes, I8), (k_scale, F32), (v_scale, F32)):
        assert a.dtype == dt and a.flags["C_CONTIGUOUS"]
    T, Hkv, D = k.shape
    num_slots = k_codes.size // (Hkv * D)
    assert k_scale.size == num_slots * Hkv and v_scale.size == num_slots * Hkv
    return _load().or_kv_write_i8(_ptr(k), _ptr(v), T, Hkv, D, _ptr(sm), _ptr(k_codes),
                                  _ptr(v_codes), _ptr(k_scale), _ptr(v_scale), num_slots)


def paged_attention_i8(q, k_codes, v_codes, k_scale, v_scale, block_table, ctx_lens,
                       page: int, scale: float | None = None):
    """INT8 KV variant of paged_attention: codes [num_blocks*page, Hkv, D],
    scales [num_blocks*page, Hkv]; returns (out [B,Hq,D], rc)."""
    q = _c(q, U16)
    k_codes = _c(k_codes, I8)
    v_codes = _c(v_codes, I8)
    k_scale = _c(k_scale, F32)
    v_scale = _c(v_scale, F32)
    bt = _c(block_table, I32)
    cl = _c(ctx_lens, I32)
    B, Hq, D = q.shape
    Hkv = k_codes.shape[-2]
    num_blocks = k_codes.size // (Hkv * D * page)
    assert k_scale.size == num_blocks * page * Hkv == v_scale.size
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    out = np.empty_like(q)
    rc = _load().or_paged_attention_i8(_ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scale),
                                       _ptr(v_scale), _ptr(bt), _ptr(cl), B, Hq, Hkv, D, page,
                                       bt.shape[1], num_blocks, scale, _ptr(out))
    return out, rc


def make_config(cfg: dict) -> Config:
    return Config(cfg["hidden"], cfg["num_q_heads"], cfg["num_kv_heads"],
                  cfg["head_dim"], cfg["intermediate"], cfg.get("num_layers", 1),
                  cfg.get("vocab", 0), cfg["page_size"], cfg.get("down_k_splits", 2),
                  cfg["rms_eps"], cfg["rope_theta"])


_WEIGHT_DTYPES = {"input_norm_w": U16, "w_qkv": I8, "s_qkv": F32, "q_norm_w": U16,
                  "k_norm_w": U16, "w_o": I8, "s_o": F32, "post_norm_w": U16,
                  "w_gate_up": I8, "s_gate_up": F32, "w_down": I8, "s_down": F32}


def _layer_struct(w: dict, keep: list) -> LayerWeights:
    s = LayerWeights()
    for name, dt in _WEIGHT_DTYPES.items():
        a = _c(w[name], dt)
        keep.append(a)
        setattr(s, name, _ptr(a))
    return s


def decode_layer(w: dict, cfg: dict, hidden, slot_mapping, block_table, ctx_lens,
                 k_cache, v_cache, taps: bool = False, k_scale=None, v_scale=None):
    """One layer; hidden [B,H] bf16 is returned updated (copy); caches updated in place.

    With k_scale and v_scale ([slots, Hkv] float32) the caches are the INT8 KV
    variant (int8 codes [slots, Hkv, D]); otherwise BF16 [slots, Hkv, D].
    Returns (hidden_out, taps_dict or None, rc)."""
    keep: list = []
    ws = _layer_struct(w, keep)
    c = make_config(cfg)
    h = _c(hidden, U16).copy()
    B, H = h.shape
    sm = _c(slot_mapping, I32)
    bt = _c(block_table, I32)
    cl = _c(ctx_lens, I32)
    assert k_cache.flags["C_CONTIGUOUS"] and v_cache.flags["C_CONTIGUOUS"]
    Hq, Hkv, D, I = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"], cfg["intermediate"]
    num_blocks = k_cache.size // (Hkv * D * cfg["page_size"])
    tap_arrays = None
    tptr = None
    if taps:
        NQ, NK = Hq * D, Hkv * D
        shapes = {
            "xn": (U16, (B, H)), "xq": (I8, (B, H)), "xs": (F32, (B,)),
            "acc_qkv": (I32, (B, NQ + 2 * NK)), "qkv": (U16, (B, NQ + 2 * NK)),
            "q_rot": (U16, (B, Hq, D)), "k_rot": (U16, (B, Hkv, D)),
            "attn": (U16, (B, NQ)), "aq": (I8, (B, NQ)), "as": (F32, (B,)),
            "acc_o": (I32, (B, H)), "h1": (U16, (B, H)), "hn": (U16, (B, H)),
            "hq": (I8, (B, H)), "hs": (F32, (B,)), "acc_gu": (I32, (B, 2 * I)),
            "act": (U16, (B, I)), "actq": (I8, (B, I)), "acts": (F32, (B,)),
            "acc_down": (I32, (B, H)),
        }
        tap_arrays = {n: np.zeros(s, dtype=dt) for n, (dt, s) in shapes.items()}
        t = LayerTaps()
        for n in TAP_NAMES:
            setattr(t, n, _ptr(tap_arrays[n]))
        tptr = ctypes.byref(t)
    if k_scale is None and v_scale is None:
        assert k_cache.dtype == U16 and v_cache.dtype == U16
        rc = _load().or_decode_layer(ctypes.byref(ws), ctypes.byref(c), B, _ptr(h), _ptr(sm),
                                     _ptr(bt), bt.shape[1], num_blocks, _ptr(cl),
                                     _ptr(k_cache), _ptr(v_cache), tptr)
    else:
        assert k_cache.dtype == I8 and v_cache.dtype == I8
        for a in (k_scale, v_scale):
            assert a.dtype == F32 and a.flags["C_CONTIGUOUS"]
            assert a.size == num_blocks * cfg["page_size"] * Hkv
        rc = _load().or_decode_layer_i8kv(ctypes.byref(ws), ctypes.byref(c), B, _ptr(h),
                                          _ptr(sm), _ptr(bt), bt.shape[1], num_blocks,
                                          _ptr(cl), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(k_scale), _ptr(v_scale), tptr)
    return h, tap_arrays, rc


def prefill_layer(w: dict, cfg: dict, hidden, slot_mapping, block_table, ctx_lens,
                  k_cache, v_cache, taps: bool = False, k_scale=None, v_scale=None):
    """One layer over a prefill chunk: M token rows, row r the token at position
    ctx_lens[r] - 1 of the sequence whose block table row it carries.

    The layer runs stage by stage over all rows (decode_layer): every row's K/V
    is written (a7) before any row attends (a8), each over its own ctx_lens[r]
    tokens, so the chunk is causal; quantisation and projections are per row.
    Hence the result equals decoding the rows one at a time in position order
    (reading of "A8W8-compatible prefill chunk": the prompt decoded as a
    chunk), which tests/test_oracle_pins.py checks."""
    return decode_layer(w, cfg, hidden, slot_mapping, block_table, ctx_lens, k_cache, v_cache,
                        taps, k_scale=k_scale, v_scale=v_scale)


def linear_bf16(x, W, residual=None) -> np.ndarray:
    """BF16 variant projection: bf16(x [M,K] . W [N,K]^T (+ residual)) -> [M,N]."""
    x = _c(x, U16)
    W = _c(W, U16)
    M, K = x.shape
    N = W.shape[0]
    assert W.shape[1] == K
    res = None if residual is None else _c(residual, U16)
    y = np.empty((M, N), U16)
    _load().or_linear_bf16(_ptr(x), M, K, _ptr(W), N, _ptr(res), _ptr(y))
    return y


def gate_up_swiglu_bf16(x, W_gu) -> np.ndarray:
    """BF16 variant Gate/Up + SwiGLU: W_gu [2I, K] -> act [M, I] (bf16)."""
    x = _c(x, U16)
    W_gu = _c(W_gu, U16)
    M, K = x.shape
    I = W_gu.shape[0] // 2
    act = np.empty((M, I), U16)
    _load().or_gate_up_swiglu_bf16(_ptr(x), M, K, _ptr(W_gu), I, _ptr(act))
    return act


BF16_TAPS = ("xn", "qkv", "q_rot", "k_rot", "attn", "h1", "hn", "act")


def decode_layer_bf16(w: dict, cfg: dict, hidden, slot_mapping, block_table, ctx_lens,
                      k_cache, v_cache, taps: bool = False):
    """BF16 (unquantised) layer; weights w hold the BF16 names of
    BF16_WEIGHT_NAMES. hidden [B,H] is returned updated (copy); the BF16 caches
    are updated in place. Returns (hidden_out, taps_dict or None, rc)."""
    keep: list = []
    ws = LayerWeightsBF16()
    for name in BF16_WEIGHT_NAMES:
        a = _c(w[name], U16)
        keep.append(a)
        setattr(ws, name, _ptr(a))
    c = make_config(cfg)
    h = _c(hidden, U16).copy()
    B, H = h.shape
    sm = _c(slot_mapping, I32)
    bt = _c(block_table, I32)
    cl = _c(ctx_lens, I32)
    assert k_cache.dtype == U16 and v_cache.dtype == U16
    assert k_cache.flags["C_CONTIGUOUS"] and v_cache.flags["C_CONTIGUOUS"]
    Hq, Hkv, D, I = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"], cfg["intermediate"]
    num_blocks = k_cache.size // (Hkv * D * cfg["page_size"])
    tap_arrays = None
    tptr = None
    if taps:
        NQ, NK = Hq * D, Hkv * D
        shapes = {"xn": (B, H), "qkv": (B, NQ + 2 * NK), "q_rot": (B, Hq, D),
                  "k_rot": (B, Hkv, D), "attn": (B, NQ), "h1": (B, H), "hn": (B, H),
                  "act": (B, I)}
        tap_arrays = {n: np.zeros(shp, dtype=U16) for n, shp in shapes.items()}
        t = LayerTaps()
        for n in BF16_TAPS:
            setattr(t, n, _ptr(tap_arrays[n]))
        tptr = ctypes.byref(t)
    rc = _load().or_decode_layer_bf16(ctypes.byref(ws), ctypes.byref(c), B, _ptr(h), _ptr(sm),
                                      _ptr(bt), bt.shape[1], num_blocks, _ptr(cl),
                                      _ptr(k_cache), _ptr(v_cache), tptr)
    return h, tap_arrays, rc


def lm_head(hn, W_lm) -> np.ndarray:
    hn = _c(hn, U16)
    W_lm = _c(W_lm, U16)
    B, H = hn.shape
    V = W_lm.shape[0]
    out = np.empty((B, V), dtype=np.float64)
    _load().or_lm_head(_ptr(hn), B, H, _ptr(W_lm), V, _ptr(out))
    return out


def argmax_f64(logits) -> np.ndarray:
    logits = _c(logits, np.float64)
    B, V = logits.shape
    out = np.empty(B, dtype=I32)
    _load().or_argmax_f64(_ptr(logits), B, V, _ptr(out))
    return out


def argmax_f32(logits) -> np.ndarray:
    logits = _c(logits, F32)
    B, V = logits.shape
    out = np.empty(B, dtype=I32)
    _load().or_argmax_f32(_ptr(logits), B, V, _ptr(out))
    return out


def decode_step(model: dict, cfg: dict, token_ids, slot_mapping, block_table, ctx_lens,
                k_caches: list, v_caches: list, want_logits: bool = False):
    """One decode step. Returns (next_tokens [B], final_hidden [B,H], logits or None, rc)."""
    keep: list = []
    L = cfg["num_layers"]
    layers = (LayerWeights * L)(*[_layer_struct(model["layers"][i], keep) for i in range(L)])
    embed = _c(model["embed"], U16)
    fnw = _c(model["final_norm_w"], U16)
    lm = _c(model["lm_head"], U16)
    m = Model(_ptr(embed), ctypes.cast(layers, _p), _ptr(fnw), _ptr(lm))
    c = make_config(cfg)
    tok = _c(token_ids, I32)
    sm = _c(slot_mapping, I32)
    bt = _c(block_table, I32)
    cl = _c(ctx_lens, I32)
    B = tok.shape[0]
    H, V = cfg["hidden"], cfg["vocab"]
    Hkv, D = cfg["num_kv_heads"], cfg["head_dim"]
    for kc, vc in zip(k_caches, v_caches):
        assert kc.flags["C_CONTIGUOUS"] and vc.flags["C_CONTIGUOUS"] and kc.dtype == U16
    num_blocks = k_caches[0].size // (Hkv * D * cfg["page_size"])
    kp = (_p * L)(*[_ptr(a) for a in k_caches])
    vp = (_p * L)(*[_ptr(a) for a in v_caches])
    nxt = np.empty(B, dtype=I32)
    fh = np.empty((B, H), dtype=U16)
    logits = np.empty((B, V), dtype=np.float64) if want_logits else None
    rc = _load().or_decode_step(ctypes.byref(m), ctypes.byref(c), B, _ptr(tok), _ptr(sm),
                                _ptr(bt), bt.shape[1], num_blocks, _ptr(cl), kp, vp,
                                _ptr(nxt), _ptr(logits), _ptr(fh))
    return nxt, fh, logits, rc
