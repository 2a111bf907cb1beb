"""Python binding of liba8w8.so, the GB300 A8W8 decode library.

Argument marshalling only: every operation runs in the CUDA kernels behind the
C ABI declared in include/a8w8.h, with the same entry-point names. PyTorch
supplies device memory and streams. BF16 tensors are passed as
``torch.bfloat16``; all tensors must be contiguous CUDA tensors.

There is no CPU fallback: if the library is missing or fails to load, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liba8w8.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "a8w8.h")

_lock = threading.Lock()
_lib = None

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_BOUNDS, ERR_WORKSPACE, ERR_CUDA = 0, -1, -2, -3, -4, -5
FLAG_PERSISTENT_STEP = 0x1
DEVERR_SLOT, DEVERR_BLOCK, DEVERR_CTX, DEVERR_TOKEN, DEVERR_POS = 0x1, 0x2, 0x4, 0x8, 0x10


class A8W8Error(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"a8w8 status {status}: {msg}")
        self.status = status


_p = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t


class Config(ctypes.Structure):
    _fields_ = [("hidden", _i), ("num_q_heads", _i), ("num_kv_heads", _i), ("head_dim", _i),
                ("intermediate", _i), ("num_layers", _i), ("vocab", _i), ("page_size", _i),
                ("down_k_splits", _i), ("rms_eps", _f), ("flags", _i)]


WEIGHT_FIELDS = ("input_norm_w", "w_qkv", "s_qkv", "q_norm_w", "k_norm_w", "w_o", "s_o",
                 "post_norm_w", "w_gate_up", "s_gate_up", "w_down", "s_down")


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, _p) for n in WEIGHT_FIELDS]


BF16_WEIGHT_FIELDS = ("input_norm_w", "w_qkv", "q_norm_w", "k_norm_w", "w_o", "post_norm_w",
                      "w_gate_up", "w_down")


class Bf16LayerWeights(ctypes.Structure):
    _fields_ = [(n, _p) for n in BF16_WEIGHT_FIELDS]


class Model(ctypes.Structure):
    _fields_ = [("embed", _p), ("layers", _p), ("final_norm_w", _p), ("lm_head", _p)]


TAP_FIELDS = ("xn", "xq", "xs", "qkv", "q_rot", "k_rot", "attn", "aq", "as", "h1", "hn", "hq",
              "hs", "act", "actq", "acts")


class LayerTaps(ctypes.Structure):
    _fields_ = [(n, _p) for n in TAP_FIELDS]


_SIGNATURES = {
    "a8w8_last_error": (ctypes.c_char_p, []),
    "a8w8_version": (_i, []),
    "a8w8_read_device_errors": (_i, [ctypes.POINTER(ctypes.c_uint), _p]),
    "a8w8_quant_rows": (_i, [_p, _i, _i, _i, _p, _p, _p]),
    "a8w8_linear": (_i, [_p, _p, _i, _i, _p, _p, _i, _i, _p, _p, _p, _p]),
    "a8w8_gate_up_swiglu": (_i, [_p, _p, _i, _i, _p, _p, _i, _p, _p, _p]),
    "a8w8_matmul_i8": (_i, [_p, _i, _i, _p, _i, _i, _i, _p, _p, _p]),
    "a8w8_rmsnorm_gate_up_swiglu": (_i, [_p, _i, _i, _p, _f, _p, _p, _i, _p, _p]),
    "paged_kv_write": (_i, [_p, _p, _i, _i, _i, _p, _p, _p, _i, _i, _p]),
    "paged_decode_attention_bf16": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _p,
                                         _p, _sz, _p]),
    "a8w8_attention_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "paged_decode_attention_bf16_noalloc": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i,
                                                 _f, _p, _p]),
    "paged_kv_write_i8": (_i, [_p, _p, _i, _i, _i, _p, _p, _p, _p, _p, _i, _i, _p]),
    "paged_decode_attention_i8kv": (_i, [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i,
                                         _f, _p, _p, _sz, _p]),
    "a8w8_decode_layer_i8kv": (_i, [_p, _p, _i, _p, _p, _p, _i, _i, _p, _p, _p, _p, _p, _p, _i,
                                    _p, _sz, _p, _p]),
    "a8w8_prefill_layer_i8kv": (_i, [_p, _p, _i, _p, _p, _p, _i, _i, _p, _p, _p, _p, _p, _p, _i,
                                     _p, _sz, _p, _p]),
    "a8w8_decode_step_i8kv": (_i, [_p, _p, _i, _p, _p, _p, _i, _i, _p, _p, _p, _p, _p, _p, _i, _p,
                                   _p, _p, _p, _sz, _p]),
    "a8w8_prefill_step": (_i, [_p, _p, _i, _p, _p, _p, _i, _i, _p, _p, _p, _p, _i, _i, _p, _p, _p,
                               _p, _sz, _p]),
    "bf16_linear": (_i, [_p, _i, _i, _p, _i, _p, _p, _p]),
    "bf16_gate_up_swiglu": (_i, [_p, _i, _i, _p, _i, _p, _p]),
    "bf16_decode_layer": (_i, [_p, _p, _i, _p, _p, _p, _i, _i, _p, _p, _p, _p, _i, _p, _sz, _p,
                               _p]),
    "a8w8_rope_table": (_i, [_p, _i, _i, ctypes.c_double, _p]),
    "a8w8_workspace_bytes": (_sz, [_p, _i, _i]),
    "a8w8_sample_workspace_bytes": (_sz, [_i, _i]),
    "a8w8_sample": (_i, [_p, _i, _i, _i, _f, _f, ctypes.c_uint64, ctypes.c_uint64, _p, _p, _sz,
                         _p]),
    "a8w8_decode_layer": (_i, [_p, _p, _i, _p, _p, _p, _i, _i, _p, _p, _p, _p, _i, _p, _sz, _p,
                               _p]),
    "a8w8_prefill_layer": (_i, [_p, _p, _i, _p, _p, _p, _i, _i, _p, _p, _p, _p, _i, _p, _sz, _p,
                                _p]),
    "a8w8_decode_step": (_i, [_p, _p, _i, _p, _p, _p, _i, _i, _p, _p, _p, _p, _i, _p, _p, _p, _p,
                              _sz, _p]),
    "a8w8_step_graph_create": (_i, [ctypes.POINTER(_p), _p, _p, _i, _i, _i, _p, _p, _p, _i, _p,
                                    _p, _p, _p, _p, _p, _p, _i, _p, _sz, _p]),
    "a8w8_step_graph_create_sampled": (_i, [ctypes.POINTER(_p), _p, _p, _i, _i, _i, _p, _p, _p,
                                            _i, _p, _p, _p, _p, _p, _p, _p, _i, _f, _f,
                                            ctypes.c_uint64, _p, _p, _sz, _p, _sz, _p]),
    "a8w8_step_graph_launch": (_i, [_p, _p]),
    "a8w8_step_graph_run_host": (_i, [_p, _p, _p, _p, _p, _p, _p]),
    "a8w8_step_graph_destroy": (None, [_p]),
}


def header_functions() -> list[str]:
    """Names of the functions include/a8w8.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return [n for n in names if n not in ("if", "while")]


def build(force: bool = False) -> str:
    from . import builder
    return builder.build(force=force)


def lib():
    """Load liba8w8.so (raises if it is missing; it is never bypassed)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise A8W8Error(ERR_CUDA, f"{LIB_PATH} is missing: run __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def last_error() -> str:
    return lib().a8w8_last_error().decode()


def _check(status: int):
    if status != OK:
        raise A8W8Error(status, last_error())


# ---------------------------------------------------------------------------
# torch plumbing
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _ptr(t):
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors"
    return t.data_ptr()


def _stream(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def make_config(cfg: dict) -> Config:
    return Config(cfg["hidden"], cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"],
                  cfg["intermediate"], cfg.get("num_layers", 1), cfg.get("vocab", 0),
                  cfg["page_size"], cfg.get("down_k_splits", 2), cfg["rms_eps"],
                  cfg.get("flags", 0))


def layer_struct(w: dict) -> LayerWeights:
    s = LayerWeights()
    for n in WEIGHT_FIELDS:
        setattr(s, n, _ptr(w[n]))
    return s


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def version() -> int:
    return lib().a8w8_version()


def read_device_errors(stream=None) -> int:
    bits = ctypes.c_uint(0)
    _check(lib().a8w8_read_device_errors(ctypes.byref(bits), _stream(stream)))
    return bits.value


def a8w8_quant_rows(x, stream=None):
    torch = _torch()
    rows, cols = x.shape
    q = torch.empty((rows, cols), dtype=torch.int8, device=x.device)
    s = torch.empty((rows,), dtype=torch.float32, device=x.device)
    _check(lib().a8w8_quant_rows(_ptr(x), rows, cols, cols, _ptr(q), _ptr(s), _stream(stream)))
    return q, s


def a8w8_linear(xq, x_scale, W, w_scale, k_splits=1, residual=None, acc_out=False, out=None,
                stream=None):
    torch = _torch()
    M, K = xq.shape
    N = W.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    acc = torch.empty((M, N), dtype=torch.int32, device=xq.device) if acc_out else None
    _check(lib().a8w8_linear(_ptr(xq), _ptr(x_scale), M, K, _ptr(W), _ptr(w_scale), N, k_splits,
                             _ptr(residual), _ptr(y), _ptr(acc), _stream(stream)))
    return (y, acc) if acc_out else y


def a8w8_gate_up_swiglu(xq, x_scale, W_gu, s_gu, acc_out=False, stream=None):
    torch = _torch()
    M, K = xq.shape
    I = W_gu.shape[0] // 2
    act = torch.empty((M, I), dtype=torch.bfloat16, device=xq.device)
    acc = torch.empty((M, 2 * I), dtype=torch.int32, device=xq.device) if acc_out else None
    _check(lib().a8w8_gate_up_swiglu(_ptr(xq), _ptr(x_scale), M, K, _ptr(W_gu), _ptr(s_gu), I,
                                     _ptr(act), _ptr(acc), _stream(stream)))
    return (act, acc) if acc_out else act


def a8w8_matmul_i8(xq, W, k0=0, k1=None, out=None, scratch=None, stream=None):
    """Exact INT32 product on the tensor cores: xq [M, K] int8 . W [N, K]^T
    over K columns [k0, k1) -> [M, N] int32. `scratch` (>= 2 M K bytes on the
    device) receives the FP16 images of xq; allocated when not given."""
    torch = _torch()
    M, K = xq.shape
    N = W.shape[0]
    k1 = K if k1 is None else k1
    acc = out if out is not None else torch.empty((M, N), dtype=torch.int32, device=xq.device)
    if scratch is None:
        scratch = torch.empty((max(M * K, 1),), dtype=torch.float16, device=xq.device)
    _check(lib().a8w8_matmul_i8(_ptr(xq), M, K, _ptr(W), N, int(k0), int(k1), _ptr(acc),
                                _ptr(scratch), _stream(stream)))
    return acc


def a8w8_rmsnorm_gate_up_swiglu(x, norm_w, eps, W_gu, s_gu, out=None, stream=None):
    """Post-attention RMSNorm + per-row quantisation + fused Gate/Up + SwiGLU
    of x [M, K] bf16 in one kernel: W_gu [2I, K] int8 -> act [M, I] bf16."""
    torch = _torch()
    M, K = x.shape
    I = W_gu.shape[0] // 2
    act = out if out is not None else torch.empty((M, I), dtype=torch.bfloat16, device=x.device)
    _check(lib().a8w8_rmsnorm_gate_up_swiglu(_ptr(x), M, K, _ptr(norm_w), float(eps), _ptr(W_gu),
                                             _ptr(s_gu), I, _ptr(act), _stream(stream)))
    return act


def paged_kv_write(k, v, slot_mapping, k_cache, v_cache, page_size, stream=None):
    T, Hkv, D = k.shape
    num_blocks = k_cache.numel() // (Hkv * D * page_size)
    _check(lib().paged_kv_write(_ptr(k), _ptr(v), T, Hkv, D, _ptr(slot_mapping), _ptr(k_cache),
                                _ptr(v_cache), num_blocks, page_size, _stream(stream)))


def attention_workspace_bytes(B, Hq, D, max_ctx) -> int:
    return lib().a8w8_attention_workspace_bytes(B, Hq, D, max_ctx)


def paged_decode_attention_bf16(q, k_cache, v_cache, block_table, ctx_lens, page_size,
                                softmax_scale=None, ws=None, out=None, stream=None):
    torch = _torch()
    B, Hq, D = q.shape
    Hkv = k_cache.shape[-2]
    num_blocks = k_cache.numel() // (Hkv * D * page_size)
    max_blocks = block_table.shape[1]
    scale = (1.0 / D ** 0.5) if softmax_scale is None else softmax_scale
    need = attention_workspace_bytes(B, Hq, D, max_blocks * page_size)
    if ws is None and need:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    o = out if out is not None else torch.empty_like(q)
    _check(lib().paged_decode_attention_bf16(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(ctx_lens), B, Hq, Hkv, D,
        page_size, max_blocks, num_blocks, scale, _ptr(o), _ptr(ws),
        0 if ws is None else ws.numel(), _stream(stream)))
    return o


NOALLOC_SCRATCH_BYTES = 8 << 20


def paged_decode_attention_bf16_noalloc(q, k_cache, v_cache, block_table, ctx_lens, page_size,
                                        softmax_scale=None, out=None, stream=None):
    """Decode attention for callers that cannot allocate device memory.

    Same result as paged_decode_attention_bf16, with the split-KV partials in
    the library's built-in 8 MiB device scratch instead of a caller workspace.
    The first call on a device looks up that scratch's address (make it before
    any stream capture); calls that overlap on the GPU share the scratch and
    race, so serialise them."""
    B, Hq, D = q.shape
    Hkv = k_cache.shape[-2]
    num_blocks = k_cache.numel() // (Hkv * D * page_size)
    scale = (1.0 / D ** 0.5) if softmax_scale is None else softmax_scale
    o = out if out is not None else _torch().empty_like(q)
    _check(lib().paged_decode_attention_bf16_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(ctx_lens), B, Hq, Hkv, D,
        page_size, block_table.shape[1], num_blocks, scale, _ptr(o), _stream(stream)))
    return o


def a8w8_rope_table(max_pos, D, theta, device="cuda", stream=None):
    torch = _torch()
    t = torch.empty((max_pos, 2 * D), dtype=torch.float32, device=device)
    _check(lib().a8w8_rope_table(_ptr(t), max_pos, D, float(theta), _stream(stream)))
    return t


def a8w8_sample(logits, temperature: float, top_p: float, seed: int, step: int, out=None,
                ws=None, stream=None):
    """Next tokens [B] int32 from logits [B, V] float32 on the device:
    temperature <= 0 is greedy; otherwise a top-p nucleus draw by the
    Gumbel-max rule with Philox4x32-10 noise keyed by (seed, step)."""
    torch = _torch()
    B, V = logits.shape
    o = out if out is not None else torch.empty(B, dtype=torch.int32, device=logits.device)
    need = lib().a8w8_sample_workspace_bytes(B, V)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=logits.device)
    _check(lib().a8w8_sample(_ptr(logits), B, V, logits.stride(0), float(temperature), float(top_p),
                             int(seed) & (2 ** 64 - 1), int(step) & (2 ** 64 - 1), _ptr(o), _ptr(ws),
                             0 if ws is None else ws.numel(), _stream(stream)))
    return o


def workspace_bytes(cfg: dict, max_B: int, max_blocks: int) -> int:
    c = make_config(cfg)
    return lib().a8w8_workspace_bytes(ctypes.byref(c), max_B, max_blocks)


def alloc_workspace(cfg: dict, max_B: int, max_blocks: int, device="cuda"):
    torch = _torch()
    return torch.empty(workspace_bytes(cfg, max_B, max_blocks), dtype=torch.uint8, device=device)


def make_taps(cfg: dict, B: int, device="cuda") -> dict:
    torch = _torch()
    H, Hq, Hkv, D, I = (cfg["hidden"], cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"],
                        cfg["intermediate"])
    bf, i8, f32 = torch.bfloat16, torch.int8, torch.float32
    shapes = {"xn": (bf, (B, H)), "hn": (bf, (B, H)), "xq": (i8, (B, H)), "xs": (f32, (B,)), "qkv": (bf, (B, (Hq + 2 * Hkv) * D)),
              "q_rot": (bf, (B, Hq, D)), "k_rot": (bf, (B, Hkv, D)), "attn": (bf, (B, Hq * D)),
              "aq": (i8, (B, Hq * D)), "as": (f32, (B,)), "h1": (bf, (B, H)),
              "hq": (i8, (B, H)), "hs": (f32, (B,)), "act": (bf, (B, I)),
              "actq": (i8, (B, I)), "acts": (f32, (B,))}
    return {n: torch.zeros(s, dtype=dt, device=device) for n, (dt, s) in shapes.items()}


def a8w8_decode_layer(weights: dict, cfg: dict, hidden, slot_mapping, block_table, ctx_lens,
                      k_cache, v_cache, rope, ws, taps: dict | None = None, stream=None):
    """One decode layer; `hidden` [B, H] bf16 is updated in place."""
    B = hidden.shape[0]
    Hkv, D, page = cfg["num_kv_heads"], cfg["head_dim"], cfg["page_size"]
    num_blocks = k_cache.numel() // (Hkv * D * page)
    c = make_config(cfg)
    w = layer_struct(weights)
    t = None
    if taps is not None:
        t = LayerTaps()
        for n in TAP_FIELDS:
            setattr(t, n, _ptr(taps.get(n)))
    _check(lib().a8w8_decode_layer(
        ctypes.byref(w), ctypes.byref(c), B, _ptr(hidden), _ptr(slot_mapping), _ptr(block_table),
        block_table.shape[1], num_blocks, _ptr(ctx_lens), _ptr(k_cache), _ptr(v_cache),
        _ptr(rope), rope.shape[0], _ptr(ws), ws.numel(),
        None if t is None else ctypes.byref(t), _stream(stream)))


def paged_kv_write_i8(k, v, slot_mapping, k_codes, v_codes, k_scale, v_scale, page_size,
                      stream=None):
    """INT8 KV variant: quantise k, v [T, Hkv, D] bf16 row by row into codes
    [slots, Hkv, D] int8 and row scales [slots, Hkv] float32."""
    T, Hkv, D = k.shape
    num_blocks = k_codes.numel() // (Hkv * D * page_size)
    _check(lib().paged_kv_write_i8(_ptr(k), _ptr(v), T, Hkv, D, _ptr(slot_mapping),
                                   _ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale),
                                   num_blocks, page_size, _stream(stream)))


def paged_decode_attention_i8kv(q, k_codes, v_codes, k_scale, v_scale, block_table, ctx_lens,
                                page_size, softmax_scale=None, ws=None, out=None, stream=None):
    """Decode attention over the INT8 KV cache (codes times row scales)."""
    torch = _torch()
    B, Hq, D = q.shape
    Hkv = k_codes.shape[-2]
    num_blocks = k_codes.numel() // (Hkv * D * page_size)
    max_blocks = block_table.shape[1]
    scale = (1.0 / D ** 0.5) if softmax_scale is None else softmax_scale
    need = attention_workspace_bytes(B, Hq, D, max_blocks * page_size)
    if ws is None and need:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    o = out if out is not None else torch.empty_like(q)
    _check(lib().paged_decode_attention_i8kv(
        _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale), _ptr(block_table),
        _ptr(ctx_lens), B, Hq, Hkv, D, page_size, max_blocks, num_blocks, scale, _ptr(o),
        _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))
    return o


def a8w8_decode_layer_i8kv(weights: dict, cfg: dict, hidden, slot_mapping, block_table, ctx_lens,
                           k_codes, v_codes, k_scale, v_scale, rope, ws,
                           taps: dict | None = None, stream=None):
    """One decode layer over an INT8 KV cache; `hidden` [B, H] bf16 is updated
    in place, the codes and row scales at the rows' slots are written."""
    B = hidden.shape[0]
    Hkv, D, page = cfg["num_kv_heads"], cfg["head_dim"], cfg["page_size"]
    num_blocks = k_codes.numel() // (Hkv * D * page)
    c = make_config(cfg)
    w = layer_struct(weights)
    t = None
    if taps is not None:
        t = LayerTaps()
        for n in TAP_FIELDS:
            setattr(t, n, _ptr(taps.get(n)))
    _check(lib().a8w8_decode_layer_i8kv(
        ctypes.byref(w), ctypes.byref(c), B, _ptr(hidden), _ptr(slot_mapping), _ptr(block_table),
        block_table.shape[1], num_blocks, _ptr(ctx_lens), _ptr(k_codes), _ptr(v_codes),
        _ptr(k_scale), _ptr(v_scale), _ptr(rope), rope.shape[0], _ptr(ws), ws.numel(),
        None if t is None else ctypes.byref(t), _stream(stream)))


def a8w8_prefill_layer_i8kv(weights: dict, cfg: dict, hidden, slot_mapping, block_table, ctx_lens,
                            k_codes, v_codes, k_scale, v_scale, rope, ws,
                            taps: dict | None = None, stream=None):
    """One layer over a prefill chunk of M rows with the INT8 KV cache (rows as
    a8w8_prefill_layer); `hidden` [M, H] bf16 is updated in place."""
    M = hidden.shape[0]
    Hkv, D, page = cfg["num_kv_heads"], cfg["head_dim"], cfg["page_size"]
    num_blocks = k_codes.numel() // (Hkv * D * page)
    c = make_config(cfg)
    w = layer_struct(weights)
    t = None
    if taps is not None:
        t = LayerTaps()
        for n in TAP_FIELDS:
            setattr(t, n, _ptr(taps.get(n)))
    _check(lib().a8w8_prefill_layer_i8kv(
        ctypes.byref(w), ctypes.byref(c), M, _ptr(hidden), _ptr(slot_mapping), _ptr(block_table),
        block_table.shape[1], num_blocks, _ptr(ctx_lens), _ptr(k_codes), _ptr(v_codes),
        _ptr(k_scale), _ptr(v_scale), _ptr(rope), rope.shape[0], _ptr(ws), ws.numel(),
        None if t is None else ctypes.byref(t), _stream(stream)))


def bf16_linear(x, W, residual=None, out=None, stream=None):
    """BF16 projection: bf16(x [M,K] . W [N,K]^T (+ residual)) -> [M, N]."""
    torch = _torch()
    M, K = x.shape
    N = W.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(lib().bf16_linear(_ptr(x), M, K, _ptr(W), N, _ptr(residual), _ptr(y), _stream(stream)))
    return y


def bf16_gate_up_swiglu(x, W_gu, stream=None):
    """BF16 fused Gate/Up + SwiGLU: W_gu [2I, K] -> act [M, I]."""
    torch = _torch()
    M, K = x.shape
    I = W_gu.shape[0] // 2
    act = torch.empty((M, I), dtype=torch.bfloat16, device=x.device)
    _check(lib().bf16_gate_up_swiglu(_ptr(x), M, K, _ptr(W_gu), I, _ptr(act), _stream(stream)))
    return act


def bf16_decode_layer(weights: dict, cfg: dict, hidden, slot_mapping, block_table, ctx_lens,
                      k_cache, v_cache, rope, ws, taps: dict | None = None, stream=None):
    """One BF16 (unquantised) decode layer; `hidden` [B, H] bf16 is updated in
    place; weights hold BF16_WEIGHT_FIELDS."""
    B = hidden.shape[0]
    Hkv, D, page = cfg["num_kv_heads"], cfg["head_dim"], cfg["page_size"]
    num_blocks = k_cache.numel() // (Hkv * D * page)
    c = make_config(cfg)
    w = Bf16LayerWeights()
    for n in BF16_WEIGHT_FIELDS:
        setattr(w, n, _ptr(weights[n]))
    t = None
    if taps is not None:
        t = LayerTaps()
        for n in TAP_FIELDS:
            setattr(t, n, _ptr(taps.get(n)))
    _check(lib().bf16_decode_layer(
        ctypes.byref(w), ctypes.byref(c), B, _ptr(hidden), _ptr(slot_mapping), _ptr(block_table),
        block_table.shape[1], num_blocks, _ptr(ctx_lens), _ptr(k_cache), _ptr(v_cache),
        _ptr(rope), rope.shape[0], _ptr(ws), ws.numel(),
        None if t is None else ctypes.byref(t), _stream(stream)))


def a8w8_prefill_layer(weights: dict, cfg: dict, hidden, slot_mapping, block_table, ctx_lens,
                       k_cache, v_cache, rope, ws, taps: dict | None = None, stream=None):
    """One layer over a prefill chunk of M token rows; `hidden` [M, H] bf16 is
    updated in place. Row r is the token at position ctx_lens[r] - 1 of the
    sequence whose block table row it carries; all rows' K/V are written
    before attention, so the chunk is causal."""
    M = hidden.shape[0]
    Hkv, D, page = cfg["num_kv_heads"], cfg["head_dim"], cfg["page_size"]
    num_blocks = k_cache.numel() // (Hkv * D * page)
    c = make_config(cfg)
    w = layer_struct(weights)
    t = None
    if taps is not None:
        t = LayerTaps()
        for n in TAP_FIELDS:
            setattr(t, n, _ptr(taps.get(n)))
    _check(lib().a8w8_prefill_layer(
        ctypes.byref(w), ctypes.byref(c), M, _ptr(hidden), _ptr(slot_mapping), _ptr(block_table),
        block_table.shape[1], num_blocks, _ptr(ctx_lens), _ptr(k_cache), _ptr(v_cache),
        _ptr(rope), rope.shape[0], _ptr(ws), ws.numel(),
        None if t is None else ctypes.byref(t), _stream(stream)))


class _ModelHandle:
    """Keeps the ctypes structs describing a model alive."""

    def __init__(self, model: dict, cfg: dict):
        L = cfg["num_layers"]
        self.layers = (LayerWeights * L)(*[layer_struct(model["layers"][i]) for i in range(L)])
        self.model = Model(_ptr(model["embed"]), ctypes.cast(self.layers, _p),
                           _ptr(model["final_norm_w"]), _ptr(model["lm_head"]))
        self.cfg = make_config(cfg)


def _cache_array(caches):
    return (_p * len(caches))(*[_ptr(c) for c in caches])


def a8w8_decode_step(model: dict, cfg: dict, token_ids, slot_mapping, block_table, ctx_lens,
                     k_caches, v_caches, rope, ws, next_tokens, logits=None, final_hidden=None,
                     stream=None):
    h = _ModelHandle(model, cfg)
    B = token_ids.shape[0]
    Hkv, D, page = cfg["num_kv_heads"], cfg["head_dim"], cfg["page_size"]
    num_blocks = k_caches[0].numel() // (Hkv * D * page)
    _check(lib().a8w8_decode_step(
        ctypes.byref(h.model), ctypes.byref(h.cfg), B, _ptr(token_ids), _ptr(slot_mapping),
        _ptr(block_table), block_table.shape[1], num_blocks, _ptr(ctx_lens),
        _cache_array(k_caches), _cache_array(v_caches), _ptr(rope), rope.shape[0],
        _ptr(next_tokens), _ptr(logits), _ptr(final_hidden), _ptr(ws), ws.numel(),
        _stream(stream)))


def a8w8_prefill_step(model: dict, cfg: dict, token_ids, slot_mapping, block_table, ctx_lens,
                      k_caches, v_caches, rope, ws, last_rows, next_tokens, logits=None,
                      stream=None):
    """The prompt rows (as a8w8_prefill_layer) through every layer, then the
    final norm, LM head and argmax on last_rows [S] -> next_tokens [S]."""
    h = _ModelHandle(model, cfg)
    M = token_ids.shape[0]
    S = last_rows.shape[0]
    Hkv, D, page = cfg["num_kv_heads"], cfg["head_dim"], cfg["page_size"]
    num_blocks = k_caches[0].numel() // (Hkv * D * page)
    _check(lib().a8w8_prefill_step(
        ctypes.byref(h.model), ctypes.byref(h.cfg), M, _ptr(token_ids), _ptr(slot_mapping),
        _ptr(block_table), block_table.shape[1], num_blocks, _ptr(ctx_lens),
        _cache_array(k_caches), _cache_array(v_caches), _ptr(rope), rope.shape[0], S,
        _ptr(last_rows), _ptr(next_tokens), _ptr(logits), _ptr(ws), ws.numel(), _stream(stream)))


def a8w8_decode_step_i8kv(model: dict, cfg: dict, token_ids, slot_mapping, block_table, ctx_lens,
                          k_codes, v_codes, k_scales, v_scales, rope, ws, next_tokens, logits=None,
                          final_hidden=None, stream=None):
    """One decode step over per-layer INT8 caches (lists of num_layers device
    tensors: codes [slots, Hkv, D] int8, row scales [slots, Hkv] float32)."""
    h = _ModelHandle(model, cfg)
    B = token_ids.shape[0]
    Hkv, D, page = cfg["num_kv_heads"], cfg["head_dim"], cfg["page_size"]
    num_blocks = k_codes[0].numel() // (Hkv * D * page)
    _check(lib().a8w8_decode_step_i8kv(
        ctypes.byref(h.model), ctypes.byref(h.cfg), B, _ptr(token_ids), _ptr(slot_mapping),
        _ptr(block_table), block_table.shape[1], num_blocks, _ptr(ctx_lens),
        _cache_array(k_codes), _cache_array(v_codes), _cache_array(k_scales),
        _cache_array(v_scales), _ptr(rope), rope.shape[0], _ptr(next_tokens), _ptr(logits),
        _ptr(final_hidden), _ptr(ws), ws.numel(), _stream(stream)))


class StepGraph:
    """A decode step captured once into a CUDA graph and replayed.

    The per-step inputs live in device tensors owned by this object:
    ``token_ids``, ``slot_mapping``, ``block_table``, ``ctx_lens`` (write them
    between replays) and ``next_tokens`` (read after a replay). With
    ``device_loop=True`` each replay also prepares the next step on the
    device (the drawn token fed back, context advanced by one token).

    ``sampling=dict(temperature=T, top_p=P, seed=S, step=s0)`` samples inside
    the graph (``a8w8_step_graph_create_sampled``): this object then owns the
    Philox step counter (``step_counter``, int64 [1], starting at s0 and
    advanced by each replay) and the sampling workspace, and ``logits`` is
    required."""

    def __init__(self, model: dict, cfg: dict, B: int, max_blocks: int, k_caches, v_caches, rope,
                 ws, logits=None, final_hidden=None, device_loop=False, stream=None,
                 sampling=None):
        torch = _torch()
        dev = k_caches[0].device
        self._h = _ModelHandle(model, cfg)
        self._keep = (model, k_caches, v_caches, rope, ws, logits, final_hidden)
        Hkv, D, page = cfg["num_kv_heads"], cfg["head_dim"], cfg["page_size"]
        num_blocks = k_caches[0].numel() // (Hkv * D * page)
        self.B, self.max_blocks = B, max_blocks
        i32 = torch.int32
        self.token_ids = torch.zeros(B, dtype=i32, device=dev)
        self.slot_mapping = torch.full((B,), -1, dtype=i32, device=dev)
        self.block_table = torch.zeros((B, max_blocks), dtype=i32, device=dev)
        self.ctx_lens = torch.zeros(B, dtype=i32, device=dev)
        self.next_tokens = torch.zeros(B, dtype=i32, device=dev)
        self._g = None
        g = _p()
        common = (ctypes.byref(g), ctypes.byref(self._h.model), ctypes.byref(self._h.cfg), B,
                  max_blocks, num_blocks, _cache_array(k_caches), _cache_array(v_caches),
                  _ptr(rope), rope.shape[0], _ptr(self.token_ids), _ptr(self.slot_mapping),
                  _ptr(self.block_table), _ptr(self.ctx_lens), _ptr(self.next_tokens),
                  _ptr(logits), _ptr(final_hidden), 1 if device_loop else 0)
        if sampling is None:
            _check(lib().a8w8_step_graph_create(*common, _ptr(ws), ws.numel(), _stream(stream)))
        else:
            if logits is None:
                raise ValueError("sampling inside the step needs a logits buffer")
            self.step_counter = torch.full((1,), int(sampling.get("step", 0)), dtype=torch.int64,
                                           device=dev)
            need = lib().a8w8_sample_workspace_bytes(B, cfg["vocab"])
            self._sample_ws = torch.empty(need, dtype=torch.uint8, device=dev)
            _check(lib().a8w8_step_graph_create_sampled(
                *common, float(sampling.get("temperature", 1.0)), float(sampling.get("top_p", 1.0)),
                int(sampling.get("seed", 0)) & (2 ** 64 - 1), _ptr(self.step_counter),
                _ptr(self._sample_ws),
                need, _ptr(ws), ws.numel(), _stream(stream)))
        self._g = g
        self._torch = torch

    def set_inputs(self, token_ids, slot_mapping, block_table, ctx_lens):
        self.token_ids.copy_(token_ids)
        self.slot_mapping.copy_(slot_mapping)
        self.block_table.copy_(block_table)
        self.ctx_lens.copy_(ctx_lens)

    def launch(self, stream=None):
        _check(lib().a8w8_step_graph_launch(self._g, _stream(stream)))

    def run_host(self, token_ids, slot_mapping, block_table, ctx_lens, next_tokens, stream=None):
        """Host (CPU, ideally pinned) int32 tensors in and out; synchronises."""
        for t in (token_ids, slot_mapping, block_table, ctx_lens, next_tokens):
            assert not t.is_cuda and t.is_contiguous() and t.dtype == self._torch.int32
        _check(lib().a8w8_step_graph_run_host(
            self._g, token_ids.data_ptr(), slot_mapping.data_ptr(), block_table.data_ptr(),
            ctx_lens.data_ptr(), next_tokens.data_ptr(), _stream(stream)))

    def close(self):
        if self._g:
            lib().a8w8_step_graph_destroy(self._g)
            self._g = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
