"""The seeded input generators: layouts that the oracle and the CUDA path both
rely on are valid (distinct pages, slots inside their request's pages, padded
rows marked), and every draw is reproducible from its seed."""
import numpy as np

import synth


def _owned_pages(bt, ctx, page):
    return [set(bt[b, :(int(c) + page - 1) // page].tolist()) for b, c in enumerate(ctx)]


def test_paged_layout_gives_each_request_its_own_pages():
    ctx = [1, 16, 17, 300, 0]
    bt, nblk = synth.paged_layout(3, ctx, 16, spare_blocks=2)
    need = [max((c + 15) // 16, 0) for c in ctx]
    assert nblk == sum(need) + 2
    assert bt.shape == (len(ctx), max(need))
    owned = _owned_pages(bt, ctx, 16)
    flat = [p for s in owned for p in s]
    assert len(flat) == len(set(flat)) == sum(need)          # no page shared
    assert all(0 <= p < nblk for p in flat)
    bt2, _ = synth.paged_layout(3, ctx, 16, spare_blocks=2)
    assert np.array_equal(bt, bt2)                            # seeded
    assert not np.array_equal(bt, synth.paged_layout(4, ctx, 16, spare_blocks=2)[0])


def test_slots_for_maps_positions_into_the_request_pages():
    ctx = [5, 40, 129]
    page = 16
    bt, _ = synth.paged_layout(5, ctx, page)
    pos = [4, 39, 128]
    sl = synth.slots_for(bt, pos, page)
    for b, p in enumerate(pos):
        assert sl[b] // page == bt[b, p // page] and sl[b] % page == p % page
    assert len(set(sl.tolist())) == len(pos)
    assert synth.slots_for(bt, [-1, 0, 3], page)[0] == -1


def test_decode_layer_case_slots_caches_and_padding():
    cfg = synth.TINY
    case = synth.decode_layer_case(cfg, 3, [16, 9, 30], seed_base=8, padded_rows=(1,))
    page = cfg["page_size"]
    bt, ctx, sl = case["block_table"], case["ctx_lens"], case["slot_mapping"]
    assert ctx.tolist() == [16, 0, 30] and sl[1] == -1
    for b in (0, 2):
        p = int(ctx[b]) - 1
        assert sl[b] == bt[b, p // page] * page + p % page
        # the decoded token's slot is still empty; the cached positions are filled
        assert not case["k_cache"][sl[b]].any()
        for t in range(p):
            s = bt[b, t // page] * page + t % page
            assert case["k_cache"][s].any() and case["v_cache"][s].any()
    assert case["hidden"].shape == (3, cfg["hidden"]) and case["hidden"].dtype == np.uint16


def test_prefill_case_rows_are_sequence_major_and_causal():
    cfg = synth.TINY
    case = synth.prefill_case(cfg, [5, 3], prior_ctx=[2, 0], seed_base=9)
    page = cfg["page_size"]
    ctx, sl, bt = case["ctx_lens"], case["slot_mapping"], case["block_table"]
    assert ctx.tolist() == [3, 4, 5, 6, 7, 1, 2, 3]
    assert len(set(sl.tolist())) == len(sl)
    seq = case["seq_block_table"]
    for r, s in enumerate([0] * 5 + [1] * 3):
        assert np.array_equal(bt[r], seq[s])
        p = int(ctx[r]) - 1
        assert sl[r] == seq[s, p // page] * page + p % page
    # the prior tokens of sequence 0 are cached, the chunk's slots are empty
    for t in range(2):
        assert case["k_cache"][seq[0, t // page] * page + t % page].any()
    assert not case["k_cache"][sl].any()


def test_batched_contexts_and_value_recipes():
    c = synth.batched_ctx_lens(11, 4096)
    assert c.min() >= 64 and c.max() <= 4096 and c.dtype == np.int32
    w = synth.int8_uniform(12, (4096,))
    assert w.min() >= -127 and w.max() <= 127
    s = synth.scales_uniform(13, 4096)
    assert s.min() >= 1e-3 and s.max() <= 4e-3
    codes, scales = synth.i8_kv_history(14, 64, 2, 16)
    assert codes.min() >= -127 and codes.max() <= 127 and scales.min() >= 2e-3
    # BF16 draws keep the float32 draw's upper 16 bits (truncation)
    x = synth.bf16_normal(15, (1000,))
    z = np.random.default_rng(15).standard_normal((1000,), dtype=np.float32)
    assert np.array_equal(x, (z.view(np.uint32) >> 16).astype(np.uint16))
