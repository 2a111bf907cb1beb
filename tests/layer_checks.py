"""Stage-by-stage parity of a decode layer (A8W8 with a BF16 or an INT8 KV
cache) against the oracle, shared by the GPU layer tests.

Every integer decision is checked bit for bit on the GPU's own inputs (the
INT8 codes and scales of each quantised row, every projection given the GPU's
quantised rows, the cache rows at their slots). Floating-point stages that the
GPU evaluates in two-float arithmetic (norms, RoPE, attention, SiLU) are held
to at most one BF16 unit of the oracle's double result and to 99.9% identical
elements; the whole layer is held to the per-layer bar.
"""
import numpy as np

import oracle
from gpu_util import (assert_layer_close, bf16_close, bf16_to_f64, bf16_ulp_diff, rel_l2,
                      to_dev, to_host)

# Share of elements of a two-float stage that must equal the oracle's BF16
# result bit for bit (the rest: one unit in the last place, at a rounding
# boundary).
STAGE_EQUAL_FRAC = 0.999


def i8_cache_case(case, seed):
    """Replace a case's BF16 caches by an INT8 history of the same slots."""
    n, Hkv, D = case["k_cache"].shape
    import synth
    kc, ks = synth.i8_kv_history(seed, n, Hkv, D)
    vc, vs = synth.i8_kv_history(seed + 1, n, Hkv, D)
    c = dict(case)
    c.update(k_cache=kc, v_cache=vc, k_scale=ks, v_scale=vs)
    return c


def run_gpu_layer(a8w8, cfg, case, with_taps=True, prefill=False):
    """The layer on the GPU; returns (hidden, taps, caches) with caches a tuple
    (k, v) for BF16 or (k_codes, v_codes, k_scale, v_scale) for INT8."""
    import torch
    i8 = "k_scale" in case
    w = {k: to_dev(v) for k, v in case["weights"].items()}
    hidden = to_dev(case["hidden"])
    caches = [to_dev(case["k_cache"]), to_dev(case["v_cache"])]
    if i8:
        caches += [to_dev(case["k_scale"]), to_dev(case["v_scale"])]
    bt = to_dev(case["block_table"])
    max_pos = int(case["block_table"].shape[1] * cfg["page_size"])
    rope = a8w8.a8w8_rope_table(max_pos, cfg["head_dim"], cfg["rope_theta"])
    ws = a8w8.alloc_workspace(cfg, hidden.shape[0], bt.shape[1])
    taps = a8w8.make_taps(cfg, hidden.shape[0]) if with_taps else None
    a8w8.read_device_errors()
    sm, cl = to_dev(case["slot_mapping"]), to_dev(case["ctx_lens"])
    if i8:
        layer = a8w8.a8w8_prefill_layer_i8kv if prefill else a8w8.a8w8_decode_layer_i8kv
        layer(w, cfg, hidden, sm, bt, cl, *caches, rope, ws, taps=taps)
    else:
        layer = a8w8.a8w8_prefill_layer if prefill else a8w8.a8w8_decode_layer
        layer(w, cfg, hidden, sm, bt, cl, *caches, rope, ws, taps=taps)
    torch.cuda.synchronize()
    assert a8w8.read_device_errors() == 0
    t = {k: to_host(v) for k, v in taps.items()} if taps else None
    return to_host(hidden), t, tuple(to_host(c) for c in caches)


def check_two_float_stage(gpu, ref, what, live=None, floor=0.1):
    """A two-float stage: every element within one BF16 unit of the oracle's
    (measured against max(|ref|, floor * RMS) for values near zero) and at
    least STAGE_EQUAL_FRAC of them identical."""
    g = gpu if live is None else gpu[live]
    r = ref if live is None else ref[live]
    if g.size == 0:
        return 1.0
    ok = bf16_close(g, r, 1, floor)
    assert ok.all(), f"{what}: {int((~ok).sum())} elements beyond one BF16 unit"
    eq = float((bf16_ulp_diff(g, r) == 0).mean())
    assert eq >= STAGE_EQUAL_FRAC, f"{what}: only {eq:.5f} of elements identical"
    return eq


def check_stages(cfg, case, out, t, caches):
    """Each stage recomputed by the oracle from the GPU's own previous stage."""
    w = case["weights"]
    i8 = "k_scale" in case
    eps, D = cfg["rms_eps"], cfg["head_dim"]
    Hq, Hkv = cfg["num_q_heads"], cfg["num_kv_heads"]
    B = case["hidden"].shape[0]
    NQ, NK = Hq * D, Hkv * D
    report = {}
    # a2: input RMSNorm (two-float vs double)
    xn = oracle.rmsnorm(case["hidden"], w["input_norm_w"], eps)
    report["xn_eq"] = check_two_float_stage(t["xn"], xn, "xn")
    # a3: quantisation of the GPU's row -- bit exact
    q, s = oracle.quant_rows(t["xn"])
    assert np.array_equal(t["xq"], q) and np.array_equal(t["xs"], s)
    # a4: QKV of the GPU's codes -- bit exact
    qkv, _ = oracle.linear(t["xq"], t["xs"], w["w_qkv"], w["s_qkv"])
    assert np.array_equal(t["qkv"], qkv)
    # a5-a6: QK norm + RoPE of the GPU's qkv
    pos = case["ctx_lens"].astype(np.int32) - 1
    live = case["ctx_lens"] > 0
    qh = oracle.rope(oracle.rmsnorm(t["qkv"][:, :NQ].reshape(B, Hq, D), w["q_norm_w"], eps),
                     np.maximum(pos, 0), cfg["rope_theta"])
    kh = oracle.rope(oracle.rmsnorm(t["qkv"][:, NQ:NQ + NK].reshape(B, Hkv, D), w["k_norm_w"], eps),
                     np.maximum(pos, 0), cfg["rope_theta"])
    report["q_rot_eq"] = check_two_float_stage(t["q_rot"], qh, "q_rot", live)
    report["k_rot_eq"] = check_two_float_stage(t["k_rot"], kh, "k_rot", live)
    # a7: the new token's K/V landed in its slot, nothing else changed
    vrow = t["qkv"][:, NQ + NK:].reshape(B, Hkv, D)
    sl_all = case["slot_mapping"]
    if i8:
        kc, vc, ks, vs = caches
        for b in range(B):
            sl = sl_all[b]
            if sl >= 0:
                kq, kss = oracle.quant_rows(t["k_rot"][b])
                vq, vss = oracle.quant_rows(vrow[b])
                assert np.array_equal(kc[sl], kq) and np.array_equal(ks[sl], kss)
                assert np.array_equal(vc[sl], vq) and np.array_equal(vs[sl], vss)
        orig = (case["k_cache"], case["v_cache"], case["k_scale"], case["v_scale"])
    else:
        kc, vc = caches
        for b in range(B):
            sl = sl_all[b]
            if sl >= 0:
                assert np.array_equal(kc[sl], t["k_rot"][b])
                assert np.array_equal(vc[sl], vrow[b])
        orig = (case["k_cache"], case["v_cache"])
    mask = np.ones(kc.shape[0], bool)
    mask[sl_all[sl_all >= 0]] = False
    for got, was in zip(caches, orig):
        assert np.array_equal(got[mask], was[mask])
    # a8: attention over the GPU's cache with the GPU's rotated q
    if i8:
        att, rc = oracle.paged_attention_i8(t["q_rot"], kc, vc, ks, vs, case["block_table"],
                                            case["ctx_lens"], cfg["page_size"])
    else:
        att, rc = oracle.paged_attention(t["q_rot"], kc, vc, case["block_table"],
                                         case["ctx_lens"], cfg["page_size"])
    assert rc == 0
    att = att.reshape(B, NQ)
    report["attn_eq"] = check_two_float_stage(t["attn"], att, "attn")
    # a9-a10: quantisation and O projection + residual -- bit exact
    aq, as_ = oracle.quant_rows(t["attn"])
    assert np.array_equal(t["aq"], aq) and np.array_equal(t["as"], as_)
    h1, _ = oracle.linear(t["aq"], t["as"], w["w_o"], w["s_o"], 1, case["hidden"])
    assert np.array_equal(t["h1"], h1)
    # a11: post-attention norm and its quantisation (exact)
    hn = oracle.rmsnorm(t["h1"], w["post_norm_w"], eps)
    report["hn_eq"] = check_two_float_stage(t["hn"], hn, "hn")
    hq, hs = oracle.quant_rows(t["hn"])
    assert np.array_equal(t["hq"], hq) and np.array_equal(t["hs"], hs)
    # a12: gate/up + SwiGLU of the GPU's codes (two-float SiLU vs double)
    act, _ = oracle.gate_up_swiglu(t["hq"], t["hs"], w["w_gate_up"], w["s_gate_up"])
    report["act_eq"] = check_two_float_stage(t["act"], act, "act", floor=1e-3)
    # a13-a14: quantisation and split-K down projection + residual -- bit exact
    dq, ds = oracle.quant_rows(t["act"])
    assert np.array_equal(t["actq"], dq) and np.array_equal(t["acts"], ds)
    o, _ = oracle.linear(t["actq"], t["acts"], w["w_down"], w["s_down"], cfg["down_k_splits"],
                         t["h1"])
    assert np.array_equal(out, o)
    return report


def stage_report(t, ot, out, ref):
    """GPU taps against the oracle's taps of the same layer: relative L2 per
    stage and the number of rows whose quantisation scale differs."""
    rep = {}
    for n in ("xn", "qkv", "attn", "h1", "hn", "act"):
        rep[n] = rel_l2(bf16_to_f64(t[n]), bf16_to_f64(ot[n]))
    for n in ("xs", "as", "hs", "acts"):
        rep[n + "_rows_differ"] = int((t[n] != ot[n]).sum())
    rep["out"] = rel_l2(bf16_to_f64(out), bf16_to_f64(ref))
    return rep


def layer_parity(a8w8, cfg, case, prefill=False):
    """Stage checks, then the whole layer against the oracle's own layer from
    the same inputs. Returns the stage report."""
    out, t, caches = run_gpu_layer(a8w8, cfg, case, prefill=prefill)
    rep = check_stages(cfg, case, out, t, caches)
    okc, ovc = case["k_cache"].copy(), case["v_cache"].copy()
    kw = {}
    if "k_scale" in case:
        kw = dict(k_scale=case["k_scale"].copy(), v_scale=case["v_scale"].copy())
    ref, ot, rc = oracle.decode_layer(case["weights"], cfg, case["hidden"], case["slot_mapping"],
                                      case["block_table"], case["ctx_lens"], okc, ovc, taps=True,
                                      **kw)
    assert rc == 0
    rep.update(stage_report(t, ot, out, ref))
    # rows where one of the four row scales differs from the oracle's: with the
    # two-float stages every BF16 value the quantiser sees equals the oracle's,
    # so none is expected; a flip would sit one BF16 unit of its absmax away
    flipped = set()
    for n in ("xs", "as", "hs", "acts"):
        for row in np.nonzero(t[n] != ot[n])[0]:
            g, o = float(t[n][row]), float(ot[n][row])
            assert abs(g - o) <= 2.0 ** -7 * abs(o) + 1e-30, (n, row, g, o)
            flipped.add(int(row))
    rep["flipped_rows"] = len(flipped)
    print("stage report:", rep)
    assert not flipped, f"rows with a quantisation scale differing from the oracle's: {sorted(flipped)}"
    assert_layer_close(out, ref, "layer output")
    # the caches the two layers wrote are identical
    if "k_scale" in case:
        for got, want in zip(caches, (okc, ovc, kw["k_scale"], kw["v_scale"])):
            assert np.array_equal(got, want)
    else:
        assert np.array_equal(caches[0], okc) and np.array_equal(caches[1], ovc)
    return rep
