"""GPU parity of the rows built beside the A8W8 decode path, each against its
pinned oracle function:

* the INT8 KV cache with FP32 row scales (the storage the pages' BF16 cache
  replaced): the quantising cache write, attention over codes times scales,
  the decode and prefill layers over it, and the decode step;
* the BF16 (unquantised) layer: its projections, fused Gate/Up + SwiGLU, and
  the whole layer;
* the prompt through the model to the first generated token.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import (STEP_REL_L2, assert_layer_close, bf16_to_f64, bf16_ulp_at, check_lm_head,
                      proj_error_bound, rel_l2, to_dev, to_host)
from layer_checks import check_two_float_stage, i8_cache_case, layer_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def a8w8():
    import w8a8_quantized_decode_gb300 as m
    m.build()
    return m


# ---------------------------------------------------------------------------
# INT8 KV cache: write
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("Hkv,D,page,nblk", [(8, 128, 128, 3), (2, 64, 16, 4)])
def test_paged_kv_write_i8_exact(a8w8, Hkv, D, page, nblk):
    T = 7
    k = synth.bf16_normal(1, (T, Hkv, D))
    v = synth.bf16_normal(2, (T, Hkv, D), std=3.0)
    k[2, 1] = 0                                  # an all-zero row: scale 0, codes 0
    v[4, 0, 5] = synth.bf16_trunc(np.float32([-3e4]))[0]   # one dominant element
    n = nblk * page
    slots = np.array([3, -1, page + 2, n - 1, 0, -1, 2 * page + 5], np.int32)
    kc, ks = synth.i8_kv_history(10, n, Hkv, D)
    vc, vs = synth.i8_kv_history(11, n, Hkv, D)
    g = [to_dev(a) for a in (kc, vc, ks, vs)]
    a8w8.read_device_errors()
    a8w8.paged_kv_write_i8(to_dev(k), to_dev(v), to_dev(slots), *g, page)
    o = [a.copy() for a in (kc, vc, ks, vs)]
    assert oracle.kv_write_i8(k, v, slots, *o) == 0
    for got, want in zip(g, o):
        assert np.array_equal(to_host(got), want)
    assert a8w8.read_device_errors() == 0


def test_paged_kv_write_i8_out_of_range_slot_is_flagged(a8w8):
    Hkv, D, page, nblk = 2, 64, 16, 2
    k = synth.bf16_normal(5, (2, Hkv, D))
    n = nblk * page
    kc = np.zeros((n, Hkv, D), np.int8)
    ks = np.zeros((n, Hkv), np.float32)
    g = [to_dev(a) for a in (kc, kc, ks, ks)]
    a8w8.read_device_errors()
    a8w8.paged_kv_write_i8(to_dev(k), to_dev(k), to_dev(np.array([5, n], np.int32)), *g, page)
    assert a8w8.read_device_errors() & a8w8.DEVERR_SLOT
    codes = to_host(g[0])
    want_q, want_s = oracle.quant_rows(k[0])
    assert np.array_equal(codes[5], want_q) and np.array_equal(to_host(g[2])[5], want_s)
    assert not np.delete(codes, 5, axis=0).any()


# ---------------------------------------------------------------------------
# INT8 KV cache: attention
# ---------------------------------------------------------------------------

I8_ATTN_CASES = [
    # B, Hq, Hkv, D, page, ctx
    (1, 40, 8, 128, 128, [256]),
    (1, 40, 8, 128, 128, [1]),
    (1, 4, 2, 64, 16, [16]),
    (4, 40, 8, 128, 128, [64, 4096, 1000, 129]),
    (3, 8, 8, 64, 16, [300, 0, 17]),
    (16, 40, 8, 128, 128, list(synth.batched_ctx_lens(5, 16))),
]


@pytest.mark.parametrize("B,Hq,Hkv,D,page,ctx", I8_ATTN_CASES)
def test_paged_attention_i8_vs_oracle(a8w8, B, Hq, Hkv, D, page, ctx):
    seed = B * 37 + D
    ctxa = np.asarray(ctx, np.int32)
    bt, nblk = synth.paged_layout(seed, np.maximum(ctxa, 1), page, spare_blocks=2)
    kc, ks = synth.i8_kv_history(seed + 1, nblk * page, Hkv, D)
    vc, vs = synth.i8_kv_history(seed + 2, nblk * page, Hkv, D)
    q = synth.bf16_normal(seed + 3, (B, Hq, D))
    a8w8.read_device_errors()
    out = a8w8.paged_decode_attention_i8kv(to_dev(q), to_dev(kc), to_dev(vc), to_dev(ks),
                                           to_dev(vs), to_dev(bt), to_dev(ctxa), page)
    ref, rc = oracle.paged_attention_i8(q, kc, vc, ks, vs, bt, ctxa, page)
    assert rc == 0
    g = to_host(out)
    for b in range(B):
        if ctxa[b] == 0:
            assert not g[b].any()
    eq = check_two_float_stage(g, ref, "INT8-KV attention")
    print("identical fraction", eq)
    assert a8w8.read_device_errors() == 0


# ---------------------------------------------------------------------------
# INT8 KV cache: decode and prefill layers
# ---------------------------------------------------------------------------

def _i8_layer(a8w8, cfg, case, seed, prefill=False):
    return layer_parity(a8w8, cfg, i8_cache_case(case, seed), prefill=prefill)


def test_i8kv_tiny_layer_b1_ctx16(a8w8):
    cfg = synth.TINY
    _i8_layer(a8w8, cfg, synth.decode_layer_case(cfg, 1, [16], seed_base=1101), 1150)


def test_i8kv_tiny_layer_b1_two_pages(a8w8):
    cfg = synth.TINY
    _i8_layer(a8w8, cfg, synth.decode_layer_case(cfg, 1, [17], seed_base=1102), 1151)


def test_i8kv_tiny_layer_batched_with_padding(a8w8):
    cfg = synth.TINY
    case = synth.decode_layer_case(cfg, 16, list(range(1, 17)), seed_base=1103,
                                   padded_rows=(3, 9))
    _i8_layer(a8w8, cfg, case, 1152)


def test_i8kv_tiny_layer_grouped_attention_long_ctx(a8w8):
    # batch x context above the grouped-attention threshold, a padded row
    cfg = synth.TINY
    ctx = [1, 17, 128, 129, 500, 1024, 1025, 1100]
    case = synth.decode_layer_case(cfg, 8, ctx, seed_base=1104, padded_rows=(2,))
    _i8_layer(a8w8, cfg, case, 1153)


def test_i8kv_qwen3_14b_layer_b1_ctx256(a8w8):
    cfg = dict(synth.QWEN3_14B, num_layers=1)
    _i8_layer(a8w8, cfg, synth.decode_layer_case(cfg, 1, [256], seed_base=1105), 1154)


def test_i8kv_qwen3_14b_layer_b16_long_ctx(a8w8):
    cfg = dict(synth.QWEN3_14B, num_layers=1)
    ctx = synth.batched_ctx_lens(1106, 16)
    case = synth.decode_layer_case(cfg, 16, list(ctx), seed_base=1106)
    _i8_layer(a8w8, cfg, case, 1155)


def test_i8kv_tiny_prefill_chunk_small(a8w8):
    cfg = synth.TINY
    case = synth.prefill_case(cfg, [7, 7, 7], prior_ctx=[0, 5, 17], seed_base=1200)
    _i8_layer(a8w8, cfg, case, 1250, prefill=True)


def test_i8kv_tiny_prefill_chunk(a8w8):
    cfg = synth.TINY
    case = synth.prefill_case(cfg, [40, 40, 40], prior_ctx=[0, 5, 17], seed_base=1201)
    _i8_layer(a8w8, cfg, case, 1251, prefill=True)


def test_i8kv_qwen3_14b_prefill_chunk(a8w8):
    cfg = dict(synth.QWEN3_14B, num_layers=1)
    case = synth.prefill_case(cfg, [40, 40], prior_ctx=[0, 130], seed_base=1202)
    _i8_layer(a8w8, cfg, case, 1252, prefill=True)


# ---------------------------------------------------------------------------
# INT8 KV cache: decode step
# ---------------------------------------------------------------------------

def _oracle_step_i8(model, cfg, tok, slots, bt, ctx, kc, vc, ks, vs):
    """The oracle's step composed from its pinned functions in the step's
    order (embedding, layers over the INT8 caches, final norm, LM head,
    argmax)."""
    h = model["embed"][np.asarray(tok)]
    for l in range(cfg["num_layers"]):
        h, _, rc = oracle.decode_layer(model["layers"][l], cfg, h, slots, bt, ctx, kc[l], vc[l],
                                       k_scale=ks[l], v_scale=vs[l])
        assert rc == 0
    fh = oracle.rmsnorm(h, model["final_norm_w"], cfg["rms_eps"])
    logits = oracle.lm_head(fh, model["lm_head"])
    return oracle.argmax_f64(logits), fh, logits


@pytest.mark.parametrize("B", [1, 3])
def test_i8kv_step_teacher_forced_vs_oracle(a8w8, B):
    import torch
    cfg = dict(synth.TINY, num_layers=2, vocab=1000)
    L, page, Hkv, D = cfg["num_layers"], cfg["page_size"], cfg["num_kv_heads"], cfg["head_dim"]
    model = synth.model_weights_host(cfg, 1300 + B)
    max_seq = 40
    max_blocks = -(-max_seq // page)
    nblk = B * max_blocks + 1
    bt = np.random.default_rng(1301 + B).permutation(nblk).astype(np.int32)[: B * max_blocks]
    bt = bt.reshape(B, max_blocks)
    n = nblk * page
    kc = [np.zeros((n, Hkv, D), np.int8) for _ in range(L)]
    vc = [np.zeros((n, Hkv, D), np.int8) for _ in range(L)]
    ks = [np.zeros((n, Hkv), np.float32) for _ in range(L)]
    vs = [np.zeros((n, Hkv), np.float32) for _ in range(L)]
    gm = dict(embed=to_dev(model["embed"]), final_norm_w=to_dev(model["final_norm_w"]),
              lm_head=to_dev(model["lm_head"]),
              layers=[{k: to_dev(v) for k, v in l.items()} for l in model["layers"]])
    g = [[to_dev(a) for a in arr] for arr in (kc, vc, ks, vs)]
    rope = a8w8.a8w8_rope_table(max_blocks * page, D, cfg["rope_theta"])
    ws = a8w8.alloc_workspace(cfg, B, max_blocks)
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    logits = torch.empty((B, cfg["vocab"]), dtype=torch.float32, device="cuda")
    fh = torch.empty((B, cfg["hidden"]), dtype=torch.bfloat16, device="cuda")
    tokens = synth.prompt_ids(1302 + B, B, cfg["vocab"])
    ctx = np.zeros(B, np.int32)
    a8w8.read_device_errors()
    for step in range(12):
        ctx = ctx + 1
        slots = synth.slots_for(bt, ctx - 1, page)
        a8w8.a8w8_decode_step_i8kv(gm, cfg, to_dev(tokens), to_dev(slots), to_dev(bt),
                                   to_dev(ctx), *g, rope, ws, nxt, logits=logits, final_hidden=fh)
        o_next, o_fh, o_logits = _oracle_step_i8(model, cfg, tokens, slots, bt, ctx, kc, vc, ks,
                                                 vs)
        g_fh = to_host(fh)
        rel = rel_l2(bf16_to_f64(g_fh), bf16_to_f64(o_fh))
        assert rel <= STEP_REL_L2, (step, rel)
        check_lm_head(g_fh, model["lm_head"], to_host(logits), to_host(nxt))
        # the caches the two sides wrote this step are identical
        for l in range(L):
            for dev_c, host_c in zip((g[0][l], g[1][l], g[2][l], g[3][l]),
                                     (kc[l], vc[l], ks[l], vs[l])):
                assert np.array_equal(to_host(dev_c), host_c), (step, l)
        tokens = o_next
    assert a8w8.read_device_errors() == 0


# ---------------------------------------------------------------------------
# BF16 (unquantised) layer
# ---------------------------------------------------------------------------

def _check_proj(gpu, ref, x, W, what, residual=False):
    """A BF16 projection with float32 sums: every element within one BF16 unit
    plus the float32 summation bound of the exact value's rounding, and at
    least 99% identical to it."""
    K = W.shape[1]
    E = proj_error_bound(x, W, K + (1 if residual else 0))
    a, b = bf16_to_f64(gpu), bf16_to_f64(ref)
    lim = bf16_ulp_at(np.maximum(np.abs(a), np.abs(b))) + E
    ok = np.abs(a - b) <= lim
    assert ok.all(), f"{what}: {int((~ok).sum())} elements beyond the bound"
    eq = float((gpu == ref).mean())
    assert eq >= 0.99, f"{what}: only {eq:.4f} identical"
    return eq


def _check_swiglu(gpu, ref, x, W_gu, what):
    """act = bf16(silu(g) u) with g, u float32 sums: one BF16 unit plus the
    first-order effect of the summation bounds of g and u."""
    I, K = W_gu.shape[0] // 2, W_gu.shape[1]
    E = proj_error_bound(x, W_gu, K)
    Eg, Eu = E[:, :I], E[:, I:]
    xf = bf16_to_f64(x)
    g = np.concatenate([xf @ bf16_to_f64(W_gu[i:min(i + 4096, I)]).T for i in range(0, I, 4096)], 1)
    u = np.concatenate([xf @ bf16_to_f64(W_gu[I + i:I + min(i + 4096, I)]).T
                        for i in range(0, I, 4096)], 1)
    a, b = bf16_to_f64(gpu), bf16_to_f64(ref)
    lim = (bf16_ulp_at(np.maximum(np.abs(a), np.abs(b))) + 1.1 * (np.abs(u) + Eu) * Eg
           + (np.abs(g) + Eg) * Eu)
    ok = np.abs(a - b) <= lim
    assert ok.all(), f"{what}: {int((~ok).sum())} elements beyond the bound"
    eq = float((gpu == ref).mean())
    assert eq >= 0.99, f"{what}: only {eq:.4f} identical"
    return eq


@pytest.mark.parametrize("M,K,N,res", [(1, 5120, 7168, False), (1, 5120, 5120, True),
                                       (1, 17408, 5120, True), (16, 5120, 5120, True),
                                       (3, 264, 40, False), (2, 17408, 153, True)])
def test_bf16_linear_vs_oracle(a8w8, M, K, N, res):
    x = synth.bf16_normal(M * 7 + K, (M, K))
    W = synth.bf16_normal(N * 3 + K, (N, K), std=0.02)
    r = synth.bf16_normal(N + 11, (M, N), std=4.0) if res else None
    y = to_host(a8w8.bf16_linear(to_dev(x), to_dev(W), residual=None if r is None else to_dev(r)))
    ref = oracle.linear_bf16(x, W, r)
    _check_proj(y, ref, x, W, "bf16_linear", res)


@pytest.mark.parametrize("M,K,I", [(1, 5120, 17408), (4, 5120, 17408), (3, 256, 512)])
def test_bf16_gate_up_swiglu_vs_oracle(a8w8, M, K, I):
    x = synth.bf16_normal(M + K, (M, K))
    W = synth.bf16_normal(I + 5, (2 * I, K), std=0.02)
    act = to_host(a8w8.bf16_gate_up_swiglu(to_dev(x), to_dev(W)))
    ref = oracle.gate_up_swiglu_bf16(x, W)
    _check_swiglu(act, ref, x, W, "bf16_gate_up_swiglu")


def _bf16_layer_parity(a8w8, cfg, case):
    import torch
    w = case["weights"]
    gw = {k: to_dev(v) for k, v in w.items()}
    hidden = to_dev(case["hidden"])
    kc, vc = to_dev(case["k_cache"]), to_dev(case["v_cache"])
    bt = to_dev(case["block_table"])
    rope = a8w8.a8w8_rope_table(case["block_table"].shape[1] * cfg["page_size"], cfg["head_dim"],
                                cfg["rope_theta"])
    B = case["hidden"].shape[0]
    ws = a8w8.alloc_workspace(cfg, B, case["block_table"].shape[1])
    taps = a8w8.make_taps(cfg, B)
    a8w8.read_device_errors()
    a8w8.bf16_decode_layer(gw, cfg, hidden, to_dev(case["slot_mapping"]), bt,
                           to_dev(case["ctx_lens"]), kc, vc, rope, ws, taps=taps)
    torch.cuda.synchronize()
    assert a8w8.read_device_errors() == 0
    t = {k: to_host(v) for k, v in taps.items()}
    out, gkc, gvc = to_host(hidden), to_host(kc), to_host(vc)
    eps, D = cfg["rms_eps"], cfg["head_dim"]
    Hq, Hkv = cfg["num_q_heads"], cfg["num_kv_heads"]
    NQ, NK = Hq * D, Hkv * D
    rep = {}
    # stage by stage, each recomputed by the oracle from the GPU's previous stage
    rep["xn"] = check_two_float_stage(t["xn"], oracle.rmsnorm(case["hidden"], w["input_norm_w"], eps),
                                      "xn")
    rep["qkv"] = _check_proj(t["qkv"], oracle.linear_bf16(t["xn"], w["w_qkv"]), t["xn"],
                             w["w_qkv"], "qkv")
    pos = np.maximum(case["ctx_lens"].astype(np.int32) - 1, 0)
    live = case["ctx_lens"] > 0
    qh = oracle.rope(oracle.rmsnorm(t["qkv"][:, :NQ].reshape(B, Hq, D), w["q_norm_w"], eps), pos,
                     cfg["rope_theta"])
    kh = oracle.rope(oracle.rmsnorm(t["qkv"][:, NQ:NQ + NK].reshape(B, Hkv, D), w["k_norm_w"], eps),
                     pos, cfg["rope_theta"])
    rep["q_rot"] = check_two_float_stage(t["q_rot"], qh, "q_rot", live)
    rep["k_rot"] = check_two_float_stage(t["k_rot"], kh, "k_rot", live)
    sl = case["slot_mapping"]
    for b in range(B):
        if sl[b] >= 0:
            assert np.array_equal(gkc[sl[b]], t["k_rot"][b])
            assert np.array_equal(gvc[sl[b]], t["qkv"][b, NQ + NK:].reshape(Hkv, D))
    att, rc = oracle.paged_attention(t["q_rot"], gkc, gvc, case["block_table"], case["ctx_lens"],
                                     cfg["page_size"])
    assert rc == 0
    rep["attn"] = check_two_float_stage(t["attn"], att.reshape(B, NQ), "attn")
    rep["h1"] = _check_proj(t["h1"], oracle.linear_bf16(t["attn"], w["w_o"], case["hidden"]),
                            t["attn"], w["w_o"], "h1", True)
    rep["hn"] = check_two_float_stage(t["hn"], oracle.rmsnorm(t["h1"], w["post_norm_w"], eps), "hn")
    rep["act"] = _check_swiglu(t["act"], oracle.gate_up_swiglu_bf16(t["hn"], w["w_gate_up"]),
                               t["hn"], w["w_gate_up"], "act")
    rep["out"] = _check_proj(out, oracle.linear_bf16(t["act"], w["w_down"], t["h1"]), t["act"],
                             w["w_down"], "out", True)
    # the whole layer against the oracle's own BF16 layer from the same inputs
    okc, ovc = case["k_cache"].copy(), case["v_cache"].copy()
    ref, _, rc = oracle.decode_layer_bf16(w, cfg, case["hidden"], sl, case["block_table"],
                                          case["ctx_lens"], okc, ovc)
    assert rc == 0
    r, m = assert_layer_close(out, ref, "BF16 layer output")
    rep.update(rel_l2=r, norm_max_abs=m, identical=float((out == ref).mean()))
    print("BF16 layer:", rep)


def _bf16_case(cfg, B, ctx, seed, padded_rows=()):
    case = synth.decode_layer_case(cfg, B, ctx, seed_base=seed, padded_rows=padded_rows)
    case["weights"] = synth.bf16_layer_weights(cfg, seed)
    return case


def test_bf16_layer_tiny_b1(a8w8):
    _bf16_layer_parity(a8w8, synth.TINY, _bf16_case(synth.TINY, 1, [16], 1400))


def test_bf16_layer_tiny_batched_with_padding(a8w8):
    _bf16_layer_parity(a8w8, synth.TINY, _bf16_case(synth.TINY, 6, [1, 5, 16, 17, 30, 9], 1401,
                                                    padded_rows=(2,)))


def test_bf16_layer_qwen3_14b_b1_ctx256(a8w8):
    cfg = dict(synth.QWEN3_14B, num_layers=1)
    _bf16_layer_parity(a8w8, cfg, _bf16_case(cfg, 1, [256], 1402))


def test_bf16_layer_qwen3_14b_b4_mixed_ctx(a8w8):
    cfg = dict(synth.QWEN3_14B, num_layers=1)
    _bf16_layer_parity(a8w8, cfg, _bf16_case(cfg, 4, [1, 77, 256, 129], 1403))


# ---------------------------------------------------------------------------
# Prompt to first token
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("prompt_lens", [[5, 9, 16], [40, 33, 27]])
def test_prefill_step_vs_oracle(a8w8, prompt_lens):
    """The prompt rows through every layer at once and the first generated
    token of each sequence, against the oracle's step over the same rows (each
    at its own position; every row's K/V is written before any row attends,
    which makes the chunk causal)."""
    import torch
    cfg = dict(synth.TINY, num_layers=2, vocab=1000)
    L, page, Hkv, D = cfg["num_layers"], cfg["page_size"], cfg["num_kv_heads"], cfg["head_dim"]
    seed = 1500 + sum(prompt_lens)
    model = synth.model_weights_host(cfg, seed)
    S = len(prompt_lens)
    bt_seq, nblk = synth.paged_layout(seed + 1, prompt_lens, page, spare_blocks=2)
    rows_bt, ctx, slots, last = [], [], [], []
    for s, n in enumerate(prompt_lens):
        for i in range(n):
            rows_bt.append(bt_seq[s])
            ctx.append(i + 1)
            slots.append(int(bt_seq[s, i // page]) * page + i % page)
        last.append(len(ctx) - 1)
    bt = np.stack(rows_bt).astype(np.int32)
    ctx = np.asarray(ctx, np.int32)
    slots = np.asarray(slots, np.int32)
    last = np.asarray(last, np.int32)
    M = len(ctx)
    tok = synth.prompt_ids(seed + 2, M, cfg["vocab"])
    n = nblk * page
    kc = [np.zeros((n, Hkv, D), np.uint16) for _ in range(L)]
    vc = [np.zeros((n, Hkv, D), np.uint16) for _ in range(L)]
    gm = dict(embed=to_dev(model["embed"]), final_norm_w=to_dev(model["final_norm_w"]),
              lm_head=to_dev(model["lm_head"]),
              layers=[{k: to_dev(v) for k, v in l.items()} for l in model["layers"]])
    gkc = [to_dev(c) for c in kc]
    gvc = [to_dev(c) for c in vc]
    rope = a8w8.a8w8_rope_table(bt.shape[1] * page, D, cfg["rope_theta"])
    ws = a8w8.alloc_workspace(cfg, M, bt.shape[1])
    nxt = torch.empty(S, dtype=torch.int32, device="cuda")
    logits = torch.empty((S, cfg["vocab"]), dtype=torch.float32, device="cuda")
    a8w8.read_device_errors()
    a8w8.a8w8_prefill_step(gm, cfg, to_dev(tok), to_dev(slots), to_dev(bt), to_dev(ctx), gkc, gvc,
                           rope, ws, to_dev(last), nxt, logits=logits)
    torch.cuda.synchronize()
    assert a8w8.read_device_errors() == 0
    o_next, o_fh, o_logits, rc = oracle.decode_step(model, cfg, tok, slots, bt, ctx, kc, vc,
                                                    want_logits=True)
    assert rc == 0
    # every layer's cache equals the oracle's (the rotated K and V of every row)
    for l in range(L):
        assert np.array_equal(to_host(gkc[l]), kc[l]), l
        assert np.array_equal(to_host(gvc[l]), vc[l]), l
    # logits of the sequences' last rows: the oracle's LM head on the oracle's
    # final hidden rows, within the float32 accumulation bound
    check_lm_head(o_fh[last], model["lm_head"], to_host(logits), to_host(nxt),
                  o_logits=o_logits[last])
