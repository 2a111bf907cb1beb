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
from gpu_util import (assert_layer_close, bf16_close, bf16_to_f64, bf16_ulp_diff, rel_l2,
                      to_dev, to_host)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def a8w8():
    import w8a8_quantized_decode_gb300 as m
    m.build()
    return m


def _run_gpu_layer(a8w8, cfg, case, with_taps=True, prefill=False):
    import torch
    w = {k: to_dev(v) for k, v in case["weights"].items()}
    hidden = to_dev(case["hidden"])
    kc, vc = to_dev(case["k_cache"]), to_dev(case["v_cache"])
    bt = to_dev(case["block_table"])
    max_pos = int(case["block_table"].shape[1] * cfg["page_size"])
    rope = a8w8.a8w8_rope_table(max_pos, cfg["head_dim"], cfg["rope_theta"])
    ws = a8w8.alloc_workspace(cfg, hidden.shape[0], bt.shape[1])
    taps = a8w8.make_taps(cfg, hidden.shape[0]) if with_taps else None
    a8w8.read_device_errors()
    layer = a8w8.a8w8_prefill_layer if prefill else a8w8.a8w8_decode_layer
    layer(w, cfg, hidden, to_dev(case["slot_mapping"]), bt, to_dev(case["ctx_lens"]), kc, vc,
          rope, ws, taps=taps)
    torch.cuda.synchronize()
    assert a8w8.read_device_errors() == 0
    t = {k: to_host(v) for k, v in taps.items()} if taps else None
    return to_host(hidden), t, to_host(kc), to_host(vc)


def _check_stages(cfg, case, out, t, kc, vc):
    """Each stage recomputed by the oracle from the GPU's own previous stage."""
    w = case["weights"]
    eps, D = cfg["rms_eps"], cfg["head_dim"]
    Hq, Hkv, I = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["intermediate"]
    B = case["hidden"].shape[0]
    NQ, NK = Hq * D, Hkv * D
    report = {}
    # a2: input RMSNorm (float32 vs double): within one BF16 ulp
    xn = oracle.rmsnorm(case["hidden"], w["input_norm_w"], eps)
    d = bf16_ulp_diff(t["xn"], xn)
    assert d.max() <= 1, d.max()
    report["xn_ulp_eq"] = float((d == 0).mean())
    # a3: quantisation of the GPU's row -- bit exact
    q, s = oracle.quant_rows(t["xn"])
    assert np.array_equal(t["xq"], q) and np.array_equal(t["xs"], s)
    # a4: QKV of the GPU's codes -- bit exact
    qkv, _ = oracle.linear(t["xq"], t["xs"], w["w_qkv"], w["s_qkv"])
    assert np.array_equal(t["qkv"], qkv)
    # a5-a6: QK norm + RoPE of the GPU's qkv (float32 vs double)
    pos = case["ctx_lens"].astype(np.int32) - 1
    live = case["ctx_lens"] > 0
    qh = oracle.rope(oracle.rmsnorm(t["qkv"][:, :NQ].reshape(B, Hq, D), w["q_norm_w"], eps),
                     np.maximum(pos, 0), cfg["rope_theta"])
    kh = oracle.rope(oracle.rmsnorm(t["qkv"][:, NQ:NQ + NK].reshape(B, Hkv, D), w["k_norm_w"], eps),
                     np.maximum(pos, 0), cfg["rope_theta"])
    # a one-ulp difference of the normalised input moves x1 cos - x2 sin by one
    # ulp of the input's scale: judged at the head's RMS scale
    assert bf16_close(t["q_rot"][live], qh[live], 2, 1.0).all()
    assert bf16_close(t["k_rot"][live], kh[live], 2, 1.0).all()
    # a7: the new token's K/V landed in its slot, nothing else changed
    for b in range(B):
        sl = case["slot_mapping"][b]
        if sl >= 0:
            assert np.array_equal(kc[sl], t["k_rot"][b])
            assert np.array_equal(vc[sl], t["qkv"][b, NQ + NK:].reshape(Hkv, D))
    mask = np.ones(kc.shape[0], bool)
    mask[case["slot_mapping"][case["slot_mapping"] >= 0]] = False
    assert np.array_equal(kc[mask], case["k_cache"][mask])
    assert np.array_equal(vc[mask], case["v_cache"][mask])
    # a8: attention over the GPU's cache with the GPU's rotated q
    att, rc = oracle.paged_attention(t["q_rot"], kc, vc, case["block_table"], case["ctx_lens"],
                                     cfg["page_size"])
    assert rc == 0
    att = att.reshape(B, NQ)
    assert rel_l2(bf16_to_f64(t["attn"]), bf16_to_f64(att)) <= 2e-3
    assert bf16_close(t["attn"], att, 2, 0.1).all()
    # a9-a10: quantisation and O projection + residual -- bit exact
    aq, as_ = oracle.quant_rows(t["attn"])
    assert np.array_equal(t["aq"], aq) and np.array_equal(t["as"], as_)
    h1, _ = oracle.linear(t["aq"], t["as"], w["w_o"], w["s_o"], 1, case["hidden"])
    assert np.array_equal(t["h1"], h1)
    # a11: post-attention norm (one ulp) and its quantisation (exact)
    hn = oracle.rmsnorm(t["h1"], w["post_norm_w"], eps)
    assert bf16_ulp_diff(t["hn"], hn).max() <= 1
    hq, hs = oracle.quant_rows(t["hn"])
    assert np.array_equal(t["hq"], hq) and np.array_equal(t["hs"], hs)
    # a12: gate/up + SwiGLU of the GPU's codes (silu float32 vs double: one ulp)
    act, _ = oracle.gate_up_swiglu(t["hq"], t["hs"], w["w_gate_up"], w["s_gate_up"])
    assert bf16_close(t["act"], act, 1, 1e-3).all()
    # a13-a14: quantisation and split-K down projection + residual -- bit exact
    dq, ds = oracle.quant_rows(t["act"])
    assert np.array_equal(t["actq"], dq) and np.array_equal(t["acts"], ds)
    o, _ = oracle.linear(t["actq"], t["acts"], w["w_down"], w["s_down"], cfg["down_k_splits"],
                         t["h1"])
    assert np.array_equal(out, o)
    return report


def _stage_report(t, ot, out, ref):
    """GPU taps against the oracle's taps of the same layer: relative L2 per
    stage and the number of rows whose quantisation scale differs."""
    rep = {}
    for n in ("xn", "qkv", "attn", "h1", "hn", "act"):
        rep[n] = rel_l2(bf16_to_f64(t[n]), bf16_to_f64(ot[n]))
    for n, on in (("xs", "xs"), ("as", "as"), ("hs", "hs"), ("acts", "acts")):
        rep[n + "_rows_differ"] = int((t[n] != ot[on]).sum())
    rep["out"] = rel_l2(bf16_to_f64(out), bf16_to_f64(ref))
    return rep


def _layer_parity(a8w8, cfg, case, max_abs_bar=None, prefill=False):
    out, t, kc, vc = _run_gpu_layer(a8w8, cfg, case, prefill=prefill)
    _check_stages(cfg, case, out, t, kc, vc)
    # whole layer against the oracle's own layer from the same inputs
    okc, ovc = case["k_cache"].copy(), case["v_cache"].copy()
    ref, ot, rc = oracle.decode_layer(case["weights"], cfg, case["hidden"], case["slot_mapping"],
                                      case["block_table"], case["ctx_lens"], okc, ovc, taps=True)
    assert rc == 0
    rep = _stage_report(t, ot, out, ref)
    print("stage report:", rep)
    # rows where one of the four row scales differs from the oracle's: each such
    # scale must sit one BF16 unit of its absmax from the oracle's
    flipped = set()
    for n in ("xs", "as", "hs", "acts"):
        for row in np.nonzero(t[n] != ot[n])[0]:
            g, o = float(t[n][row]), float(ot[n][row])
            assert abs(g - o) <= 2.0 ** -7 * abs(o) + 1e-30, (n, row, g, o)
            flipped.add(int(row))
    assert len(flipped) <= max(1, len(t["xs"]) // 8), f"too many rows with a flipped scale: {flipped}"
    try:
        return assert_layer_close(out, ref, "layer output", sorted(flipped), max_abs_bar)
    except AssertionError as e:
        raise AssertionError(f"{e}; stages {rep}") from None


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
    # Batch 16 with contexts up to 4096 (grouped attention, tensor-core
    # projections). Every stage is bit-exact on the GPU's own inputs (checked
    # above); should a BF16 rounding ever differ from the oracle's, one flipped
    # act code moves a down-projection output by |W| * s_act * s_w, up to ~9%
    # of the RMS, hence the max-abs bar of 0.15 of the RMS for this case.
    cfg = dict(synth.QWEN3_14B, num_layers=1)
    ctx = synth.batched_ctx_lens(106, 16)
    case = synth.decode_layer_case(cfg, 16, list(ctx), seed_base=106)
    _layer_parity(a8w8, cfg, case, max_abs_bar=0.15)


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
