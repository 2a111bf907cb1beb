"""GPU parity of the fused decode layer against the oracle.

Stage by stage (through the layer's taps), every integer decision is checked
bit for bit on the GPU's own inputs: the INT8 codes and scales of each
quantised row, and every projection output given the GPU's quantised rows.
Floating-point stages are checked against the oracle within a few BF16 units,
and the whole layer against the oracle's layer at the stated bar.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import bf16_to_f64, rel_l2, to_dev, to_host
from layer_checks import layer_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def a8w8():
    import w8a8_quantized_decode_gb300 as m
    m.build()
    return m


def _layer_parity(a8w8, cfg, case, prefill=False):
    return layer_parity(a8w8, cfg, case, prefill=prefill)


def test_tiny_layer_b1_ctx16(a8w8):
    # 16 tokens in one 16-token page, the decoded token included
    cfg = synth.TINY
    _layer_parity(a8w8, cfg, synth.decode_layer_case(cfg, 1, [16], seed_base=101))


def test_tiny_layer_b1_two_pages(a8w8):
    # 16 cached tokens plus the decoded one at position 16, on a second page
    cfg = synth.TINY
    _layer_parity(a8w8, cfg, synth.decode_layer_case(cfg, 1, [17], seed_base=102))


def test_tiny_layer_batched_with_padding(a8w8):
    cfg = synth.TINY
    case = synth.decode_layer_case(cfg, 16, list(range(1, 17)), seed_base=103, padded_rows=(3, 9))
    _layer_parity(a8w8, cfg, case)


def test_qwen3_14b_layer_b1_ctx256(a8w8):
    cfg = dict(synth.QWEN3_14B, num_layers=1)
    _layer_parity(a8w8, cfg, synth.decode_layer_case(cfg, 1, [256], seed_base=104))


def test_qwen3_14b_layer_b4_mixed_ctx(a8w8):
    cfg = dict(synth.QWEN3_14B, num_layers=1)
    case = synth.decode_layer_case(cfg, 4, [1, 77, 256, 129], seed_base=105)
    _layer_parity(a8w8, cfg, case)


def test_qwen3_14b_layer_b16_long_ctx(a8w8):
    # batch 16 with contexts up to 4096 (grouped attention, tensor-core
    # projections), held to the same per-layer bar as every other case
    cfg = dict(synth.QWEN3_14B, num_layers=1)
    ctx = synth.batched_ctx_lens(106, 16)
    case = synth.decode_layer_case(cfg, 16, list(ctx), seed_base=106)
    _layer_parity(a8w8, cfg, case)


def test_tiny_layer_grouped_attention_long_ctx(a8w8):
    # batch x context above the grouped-attention threshold: one CTA per (row,
    # KV head, 128-token chunk); contexts of one token, exactly one chunk, one
    # chunk and a token, and nine chunks, and a padded row
    cfg = synth.TINY
    ctx = [1, 17, 128, 129, 500, 1024, 1025, 1100]
    case = synth.decode_layer_case(cfg, 8, ctx, seed_base=107, padded_rows=(2,))
    _layer_parity(a8w8, cfg, case)


def test_qwen3_14b_layer_grouped_attention_b2(a8w8):
    # two rows, 4096 and 2049 tokens: 33 and 17 chunks merged in the kernel
    cfg = dict(synth.QWEN3_14B, num_layers=1)
    case = synth.decode_layer_case(cfg, 2, [4096, 2049], seed_base=108)
    _layer_parity(a8w8, cfg, case)


# ---------------------------------------------------------------------------
# Prefill chunk: M token rows through the layer at once (causal by ctx_lens)
# ---------------------------------------------------------------------------

def test_tiny_prefill_chunk_small(a8w8):
    # three sequences of 7 new tokens after 0, 5 and 17 cached ones (21 rows:
    # the 16-row tensor-core projections)
    cfg = synth.TINY
    case = synth.prefill_case(cfg, [7, 7, 7], prior_ctx=[0, 5, 17], seed_base=200)
    _layer_parity(a8w8, cfg, case, prefill=True)


def test_tiny_prefill_chunk(a8w8):
    # three sequences of 40 new tokens after 0, 5 and 17 cached ones (120 rows:
    # the tiled GEMM, a partial 128-row tile)
    cfg = synth.TINY
    case = synth.prefill_case(cfg, [40, 40, 40], prior_ctx=[0, 5, 17], seed_base=201)
    _layer_parity(a8w8, cfg, case, prefill=True)


def test_qwen3_14b_prefill_chunk(a8w8):
    # 80 rows through the tiled GEMM at the Qwen3-14B shapes
    cfg = dict(synth.QWEN3_14B, num_layers=1)
    case = synth.prefill_case(cfg, [40, 40], prior_ctx=[0, 130], seed_base=202)
    _layer_parity(a8w8, cfg, case, prefill=True)


@pytest.mark.slow
def test_qwen3_14b_prefill_4x512_vs_oracle(a8w8):
    # the pages' prefill-chunk workload at full size (4 sequences x 512 tokens,
    # M = 2048, the tiled GEMM and the grouped attention) against the oracle's
    # layer over the same chunk, stage by stage and as a whole
    cfg = dict(synth.QWEN3_14B, num_layers=1)
    case = synth.prefill_case(cfg, [512] * 4, seed_base=203)
    _layer_parity(a8w8, cfg, case, prefill=True)


def test_qwen3_14b_prefill_4x512_equals_sequential_decode(a8w8):
    # the pages' prefill-chunk workload (4 sequences x 512 tokens, M = 2048):
    # the chunk through the prefill entry against the same rows decoded one
    # position at a time (4 rows per call) on the GPU; both write the caches
    import torch
    cfg = dict(synth.QWEN3_14B, num_layers=1)
    case = synth.prefill_case(cfg, [512] * 4, seed_base=203)
    w = {k: to_dev(v) for k, v in case["weights"].items()}
    bt_rows = to_dev(case["block_table"])
    nb = case["block_table"].shape[1]
    rope = a8w8.a8w8_rope_table(nb * cfg["page_size"], cfg["head_dim"], cfg["rope_theta"])
    h1 = to_dev(case["hidden"])
    kc1, vc1 = to_dev(case["k_cache"]), to_dev(case["v_cache"])
    ws = a8w8.alloc_workspace(cfg, 2048, nb)
    a8w8.read_device_errors()
    a8w8.a8w8_prefill_layer(w, cfg, h1, to_dev(case["slot_mapping"]), bt_rows,
                            to_dev(case["ctx_lens"]), kc1, vc1, rope, ws)
    torch.cuda.synchronize()
    assert a8w8.read_device_errors() == 0
    h2 = to_dev(case["hidden"])
    kc2, vc2 = to_dev(case["k_cache"]), to_dev(case["v_cache"])
    ws4 = a8w8.alloc_workspace(cfg, 4, nb)
    slots, ctx = to_dev(case["slot_mapping"]), to_dev(case["ctx_lens"])
    for i in range(512):
        rows = torch.arange(4, device=h2.device) * 512 + i
        hb = h2[rows].contiguous()
        a8w8.a8w8_decode_layer(w, cfg, hb, slots[rows].contiguous(), bt_rows[rows].contiguous(),
                               ctx[rows].contiguous(), kc2, vc2, rope, ws4)
        h2[rows] = hb
    torch.cuda.synchronize()
    assert a8w8.read_device_errors() == 0
    a, b = to_host(h1), to_host(h2)
    same = (a == b).mean()
    print("prefill vs sequential decode: identical fraction", same)
    assert same >= 0.999, same
    assert rel_l2(bf16_to_f64(a), bf16_to_f64(b)) <= 5e-3
    assert (to_host(kc1) == to_host(kc2)).mean() >= 0.9999
    assert (to_host(vc1) == to_host(vc2)).mean() == 1.0
