"""Seeded synthetic inputs for the A8W8 decode workloads.

This module only draws random numbers and lays them out; it holds none of the
decode method's arithmetic. Both the CPU oracle and the CUDA path are fed from
it, which is the only thing the two sides share.

Distributions (one generator per tensor, seeded ``seed_base + tensor_id``):
  * INT8 weights: integers uniform in [-127, 127];
  * FP32 per-output-channel weight scales: uniform in [1e-3, 4e-3];
  * norm weights: BF16 1 + N(0, 0.02);
  * hidden states, cached K/V, embeddings: BF16 N(0, 1);
  * LM head: BF16 N(0, 0.02^2);
  * BF16 (unquantised) layer projections: BF16 N(0, 0.02^2);
  * INT8 KV history: codes uniform in [-127, 127], FP32 row scales uniform in
    [2e-3, 3e-2].
BF16 values are made by keeping the upper 16 bits of a float32 draw (a
truncation, so no rounding rule of the method is involved).

Two generators exist: numpy on the host (tests, small and single-layer
workloads) and torch on the device (the 40-layer workloads, whose 13 GB of
weights are too slow to draw on the host). For the same seed they give
different values; each workload states which one it used.
"""
from __future__ import annotations

import math

import numpy as np

# --------------------------------------------------------------------------
# Workload shapes
# --------------------------------------------------------------------------

TINY = dict(name="tiny_layer_b1", hidden=256, num_q_heads=4, num_kv_heads=2,
            head_dim=64, intermediate=512, num_layers=1, vocab=0, page_size=16,
            down_k_splits=2, rms_eps=1e-6, rope_theta=1e6)

QWEN3_14B = dict(name="qwen3_14b", hidden=5120, num_q_heads=40, num_kv_heads=8,
                 head_dim=128, intermediate=17408, num_layers=40, vocab=151936,
                 page_size=128, down_k_splits=2, rms_eps=1e-6, rope_theta=1e6)

WEIGHT_NAMES = ("input_norm_w", "w_qkv", "s_qkv", "q_norm_w", "k_norm_w", "w_o",
                "s_o", "post_norm_w", "w_gate_up", "s_gate_up", "w_down", "s_down")


def with_layers(cfg: dict, num_layers: int) -> dict:
    c = dict(cfg)
    c["num_layers"] = num_layers
    return c


def weight_shapes(cfg: dict) -> dict:
    H, Hq, Hkv, D, I = (cfg["hidden"], cfg["num_q_heads"], cfg["num_kv_heads"],
                        cfg["head_dim"], cfg["intermediate"])
    nqkv = Hq * D + 2 * Hkv * D
    return {
        "input_norm_w": ("bf16", (H,)), "w_qkv": ("i8", (nqkv, H)), "s_qkv": ("f32", (nqkv,)),
        "q_norm_w": ("bf16", (D,)), "k_norm_w": ("bf16", (D,)),
        "w_o": ("i8", (H, Hq * D)), "s_o": ("f32", (H,)),
        "post_norm_w": ("bf16", (H,)),
        "w_gate_up": ("i8", (2 * I, H)), "s_gate_up": ("f32", (2 * I,)),
        "w_down": ("i8", (H, I)), "s_down": ("f32", (H,)),
    }


def layer_weight_bytes(cfg: dict) -> int:
    """Bytes of one layer's weights (INT8 matrices, FP32 scales, BF16 norms)."""
    size = {"bf16": 2, "i8": 1, "f32": 4}
    return sum(size[k] * math.prod(s) for k, s in weight_shapes(cfg).values())


# --------------------------------------------------------------------------
# Host (numpy) generators
# --------------------------------------------------------------------------

def _rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def bf16_trunc(f: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values, as uint16 BF16 bit patterns."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def bf16_normal(seed: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    z = _rng(seed).standard_normal(shape, dtype=np.float32)
    return bf16_trunc(z * np.float32(std) + np.float32(mean))


def int8_uniform(seed: int, shape) -> np.ndarray:
    return _rng(seed).integers(-127, 128, size=shape, dtype=np.int8)


def scales_uniform(seed: int, n: int) -> np.ndarray:
    return _rng(seed).uniform(1e-3, 4e-3, size=n).astype(np.float32)


def layer_weights(cfg: dict, seed_base: int, layer: int = 0) -> dict:
    """One layer's weights as numpy arrays (BF16 as uint16)."""
    out = {}
    for i, (name, (kind, shape)) in enumerate(weight_shapes(cfg).items()):
        seed = seed_base + 1000 * (layer + 1) + i
        if kind == "i8":
            out[name] = int8_uniform(seed, shape)
        elif kind == "f32":
            out[name] = scales_uniform(seed, shape[0])
        else:
            out[name] = bf16_normal(seed, shape, mean=1.0, std=0.02)
    return out


def bf16_layer_weights(cfg: dict, seed_base: int, layer: int = 0) -> dict:
    """One BF16 (unquantised) layer's weights: the A8W8 layer's matrices in
    BF16 N(0, 0.02^2), norm weights as there, no scales."""
    out = {}
    for i, (name, (kind, shape)) in enumerate(weight_shapes(cfg).items()):
        seed = seed_base + 1000 * (layer + 1) + 500 + i
        if kind == "i8":
            out[name] = bf16_normal(seed, shape, std=0.02)
        elif kind == "bf16":
            out[name] = bf16_normal(seed, shape, mean=1.0, std=0.02)
    return out


def i8_kv_history(seed: int, num_slots: int, Hkv: int, D: int):
    """Random INT8 KV cache contents: codes [slots, Hkv, D], scales [slots, Hkv]."""
    g = _rng(seed)
    codes = g.integers(-127, 128, size=(num_slots, Hkv, D), dtype=np.int8)
    scales = g.uniform(2e-3, 3e-2, size=(num_slots, Hkv)).astype(np.float32)
    return codes, scales


def hidden_states(seed: int, B: int, H: int) -> np.ndarray:
    return bf16_normal(seed, (B, H))


def paged_layout(seed: int, ctx_lens, page: int, extra_tokens: int = 0,
                 spare_blocks: int = 0):
    """Block tables filled from a seeded permutation of the physical pages.

    Request b owns ceil((ctx_lens[b] + extra_tokens) / page) pages. Returns
    (block_table [B, max_blocks] int32, num_blocks). Unused table entries are 0.
    """
    ctx_lens = np.asarray(ctx_lens, dtype=np.int64)
    need = [int(math.ceil((c + extra_tokens) / page)) for c in ctx_lens]
    total = sum(need) + spare_blocks
    perm = _rng(seed).permutation(total).astype(np.int32)
    max_blocks = max(max(need), 1)
    bt = np.zeros((len(ctx_lens), max_blocks), dtype=np.int32)
    o = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[o:o + n]
        o += n
    return bt, total


def slots_for(block_table: np.ndarray, positions, page: int) -> np.ndarray:
    """Cache slot of each request's token at `positions[b]` (-1 where < 0)."""
    out = np.empty(len(positions), dtype=np.int32)
    for b, p in enumerate(positions):
        p = int(p)
        out[b] = -1 if p < 0 else int(block_table[b, p // page]) * page + p % page
    return out


def kv_cache(seed: int, num_blocks: int, page: int, Hkv: int, D: int,
             block_table=None, ctx_lens=None) -> np.ndarray:
    """A [num_blocks*page, Hkv, D] BF16 cache with N(0,1) entries.

    When a block table and the context lengths are given, only the cached
    positions of each request are filled; every other slot is zero."""
    full = bf16_normal(seed, (num_blocks * page, Hkv, D))
    if block_table is None:
        return full
    cache = np.zeros_like(full)
    for b, n in enumerate(ctx_lens):
        for t in range(int(n)):
            s = int(block_table[b, t // page]) * page + t % page
            cache[s] = full[s]
    return cache


def decode_layer_case(cfg: dict, B: int, ctx_lens, seed_base: int = 1234,
                      spare_blocks: int = 1, padded_rows=()):
    """Inputs of one decode layer: weights, hidden, paged caches and tables.

    ctx_lens counts the decoded token (its position is ctx_len - 1, its K/V go
    to that position's slot). Cached positions 0..ctx_len-2 hold N(0,1) K/V.
    Rows listed in padded_rows get ctx_len 0 and slot -1."""
    ctx = np.asarray(ctx_lens, dtype=np.int32).copy()
    page = cfg["page_size"]
    bt, nblk = paged_layout(seed_base + 7, np.maximum(ctx, 1), page,
                            spare_blocks=spare_blocks)
    for r in padded_rows:
        ctx[r] = 0
    pos = ctx.astype(np.int64) - 1
    slots = slots_for(bt, pos, page)
    cached = np.maximum(ctx - 1, 0)
    Hkv, D = cfg["num_kv_heads"], cfg["head_dim"]
    kc = kv_cache(seed_base + 8, nblk, page, Hkv, D, bt, cached)
    vc = kv_cache(seed_base + 9, nblk, page, Hkv, D, bt, cached)
    return dict(
        weights=layer_weights(cfg, seed_base),
        hidden=hidden_states(seed_base + 5, B, cfg["hidden"]),
        ctx_lens=ctx, slot_mapping=slots, block_table=bt, num_blocks=nblk,
        k_cache=kc, v_cache=vc)


def prefill_case(cfg: dict, seq_lens, prior_ctx=None, seed_base: int = 4321,
                 spare_blocks: int = 1):
    """Inputs of one layer over a prefill chunk: sequences s = 0.. with
    seq_lens[s] new tokens after prior_ctx[s] cached ones (N(0,1) K/V).

    Rows are sequence-major; row (s, i) is the token at position
    prior_ctx[s] + i, carries its sequence's block table row, ctx_len
    prior_ctx[s] + i + 1 and the slot of that position."""
    seq_lens = [int(n) for n in seq_lens]
    prior = [0] * len(seq_lens) if prior_ctx is None else [int(c) for c in prior_ctx]
    page = cfg["page_size"]
    bt_seq, nblk = paged_layout(seed_base + 7, [p + n for p, n in zip(prior, seq_lens)], page,
                                spare_blocks=spare_blocks)
    rows_bt, ctx, slots = [], [], []
    for s, (p, n) in enumerate(zip(prior, seq_lens)):
        for i in range(n):
            pos = p + i
            rows_bt.append(bt_seq[s])
            ctx.append(pos + 1)
            slots.append(int(bt_seq[s, pos // page]) * page + pos % page)
    bt = np.stack(rows_bt).astype(np.int32)
    Hkv, D = cfg["num_kv_heads"], cfg["head_dim"]
    kc = kv_cache(seed_base + 8, nblk, page, Hkv, D, bt_seq, prior)
    vc = kv_cache(seed_base + 9, nblk, page, Hkv, D, bt_seq, prior)
    M = len(ctx)
    return dict(
        weights=layer_weights(cfg, seed_base),
        hidden=hidden_states(seed_base + 5, M, cfg["hidden"]),
        ctx_lens=np.asarray(ctx, np.int32), slot_mapping=np.asarray(slots, np.int32),
        block_table=bt, num_blocks=nblk, k_cache=kc, v_cache=vc,
        seq_block_table=bt_seq, prior_ctx=np.asarray(prior, np.int32),
        seq_lens=np.asarray(seq_lens, np.int32))


def model_weights_host(cfg: dict, seed_base: int) -> dict:
    """A whole model on the host (small configs only)."""
    H, V = cfg["hidden"], cfg["vocab"]
    return dict(
        embed=bf16_normal(seed_base + 11, (V, H)),
        layers=[layer_weights(cfg, seed_base, l) for l in range(cfg["num_layers"])],
        final_norm_w=bf16_normal(seed_base + 12, (H,), mean=1.0, std=0.02),
        lm_head=bf16_normal(seed_base + 13, (V, H), std=0.02),
    )


def prompt_ids(seed: int, n: int, vocab: int) -> np.ndarray:
    return _rng(seed).integers(0, vocab, size=n).astype(np.int32)


def batched_ctx_lens(seed: int, B: int, lo: int = 64, hi: int = 4096) -> np.ndarray:
    """Per-request context lengths uniform in [lo, hi]."""
    return _rng(seed).integers(lo, hi + 1, size=B).astype(np.int32)


# --------------------------------------------------------------------------
# Device (torch) generators, for the 40-layer workloads
# --------------------------------------------------------------------------

def _torch_gen(seed: int, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def t_bf16_normal(seed: int, shape, device, mean: float = 0.0, std: float = 1.0):
    import torch
    z = torch.randn(shape, dtype=torch.float32, device=device,
                    generator=_torch_gen(seed, device))
    if std != 1.0:
        z.mul_(std)
    if mean != 0.0:
        z.add_(mean)
    return (z.view(torch.int32) >> 16).to(torch.int16).view(torch.bfloat16)


def t_int8_uniform(seed: int, shape, device):
    import torch
    return torch.randint(-127, 128, shape, dtype=torch.int8, device=device,
                         generator=_torch_gen(seed, device))


def t_scales_uniform(seed: int, n: int, device):
    import torch
    u = torch.rand(n, dtype=torch.float32, device=device, generator=_torch_gen(seed, device))
    return u.mul_(3e-3).add_(1e-3)


def t_layer_weights(cfg: dict, seed_base: int, layer: int, device) -> dict:
    out = {}
    for i, (name, (kind, shape)) in enumerate(weight_shapes(cfg).items()):
        seed = seed_base + 1000 * (layer + 1) + i
        if kind == "i8":
            out[name] = t_int8_uniform(seed, shape, device)
        elif kind == "f32":
            out[name] = t_scales_uniform(seed, shape[0], device)
        else:
            out[name] = t_bf16_normal(seed, shape, device, mean=1.0, std=0.02)
    return out


def t_bf16_layer_weights(cfg: dict, seed_base: int, layer: int, device) -> dict:
    """Device draw of one BF16 (unquantised) layer's weights (as
    bf16_layer_weights: matrices N(0, 0.02^2), norm weights 1 + N(0, 0.02))."""
    out = {}
    for i, (name, (kind, shape)) in enumerate(weight_shapes(cfg).items()):
        seed = seed_base + 1000 * (layer + 1) + 500 + i
        if kind == "i8":
            out[name] = t_bf16_normal(seed, shape, device, std=0.02)
        elif kind == "bf16":
            out[name] = t_bf16_normal(seed, shape, device, mean=1.0, std=0.02)
    return out


def t_i8_kv_history(seed: int, num_slots: int, Hkv: int, D: int, device):
    """Device draw of INT8 KV cache contents (as i8_kv_history)."""
    import torch
    codes = torch.randint(-127, 128, (num_slots, Hkv, D), dtype=torch.int8, device=device,
                          generator=_torch_gen(seed, device))
    u = torch.rand((num_slots, Hkv), dtype=torch.float32, device=device,
                   generator=_torch_gen(seed + 1, device))
    return codes, u.mul_(2.8e-2).add_(2e-3)


def t_model_weights(cfg: dict, seed_base: int, device) -> dict:
    H, V = cfg["hidden"], cfg["vocab"]
    return dict(
        embed=t_bf16_normal(seed_base + 11, (V, H), device),
        layers=[t_layer_weights(cfg, seed_base, l, device) for l in range(cfg["num_layers"])],
        final_norm_w=t_bf16_normal(seed_base + 12, (H,), device, mean=1.0, std=0.02),
        lm_head=t_bf16_normal(seed_base + 13, (V, H), device, std=0.02),
    )
