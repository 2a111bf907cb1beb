"""GPU parity of the decode step (embedding, layers, final norm, LM head,
greedy argmax) against the oracle, plus the replayable graph and the
host-buffer entry point."""
import numpy as np
import pytest

import oracle
import synth
from oracle import sampling
from gpu_util import STEP_REL_L2, bf16_to_f64, check_lm_head, rel_l2, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def a8w8():
    import w8a8_quantized_decode_gb300 as m
    m.build()
    return m


class Session:
    """A small decode session: host model + caches, mirrored on the GPU."""

    def __init__(self, a8w8, cfg, B, max_seq, seed):
        import torch
        self.a8w8, self.cfg, self.B = a8w8, cfg, B
        self.page = cfg["page_size"]
        self.max_blocks = -(-max_seq // self.page)
        self.model = synth.model_weights_host(cfg, seed)
        nblk = B * self.max_blocks + 1
        perm = np.random.default_rng(seed + 1).permutation(nblk).astype(np.int32)
        self.bt = perm[: B * self.max_blocks].reshape(B, self.max_blocks)
        self.nblk = nblk
        Hkv, D = cfg["num_kv_heads"], cfg["head_dim"]
        L = cfg["num_layers"]
        self.kc = [np.zeros((nblk * self.page, Hkv, D), np.uint16) for _ in range(L)]
        self.vc = [np.zeros((nblk * self.page, Hkv, D), np.uint16) for _ in range(L)]
        self.gm = dict(embed=to_dev(self.model["embed"]), final_norm_w=to_dev(self.model["final_norm_w"]),
                       lm_head=to_dev(self.model["lm_head"]),
                       layers=[{k: to_dev(v) for k, v in l.items()} for l in self.model["layers"]])
        self.gkc = [to_dev(c) for c in self.kc]
        self.gvc = [to_dev(c) for c in self.vc]
        self.rope = a8w8.a8w8_rope_table(self.max_blocks * self.page, D, cfg["rope_theta"])
        self.ws = a8w8.alloc_workspace(cfg, B, self.max_blocks)
        self.next = torch.empty(B, dtype=torch.int32, device="cuda")
        self.logits = torch.empty((B, cfg["vocab"]), dtype=torch.float32, device="cuda")
        self.fh = torch.empty((B, cfg["hidden"]), dtype=torch.bfloat16, device="cuda")
        self.ctx = np.zeros(B, np.int32)

    def inputs(self, tokens):
        ctx = self.ctx + 1
        slots = synth.slots_for(self.bt, ctx - 1, self.page)
        return np.asarray(tokens, np.int32), slots, ctx

    def step_both(self, tokens):
        """One step on both sides with the same tokens; returns the comparison."""
        tok, slots, ctx = self.inputs(tokens)
        self.a8w8.a8w8_decode_step(self.gm, self.cfg, to_dev(tok), to_dev(slots), to_dev(self.bt),
                                   to_dev(ctx), self.gkc, self.gvc, self.rope, self.ws, self.next,
                                   logits=self.logits, final_hidden=self.fh)
        o_next, o_fh, o_logits, rc = oracle.decode_step(self.model, self.cfg, tok, slots, self.bt,
                                                        ctx, self.kc, self.vc, want_logits=True)
        assert rc == 0
        self.ctx = ctx
        g_fh = to_host(self.fh)
        g_logits = to_host(self.logits)
        g_next = to_host(self.next)
        return dict(rel=rel_l2(bf16_to_f64(g_fh), bf16_to_f64(o_fh)), g_next=g_next, o_next=o_next,
                    g_logits=g_logits, o_logits=o_logits, g_fh=g_fh)


@pytest.mark.parametrize("B", [1, 3, 6])
def test_step_teacher_forced_vs_oracle(a8w8, B):
    cfg = dict(synth.TINY, num_layers=3, vocab=4099)
    s = Session(a8w8, cfg, B, max_seq=40, seed=200 + B)
    tokens = synth.prompt_ids(300 + B, B, cfg["vocab"])
    agree = []
    for step in range(20):
        r = s.step_both(tokens)
        assert r["rel"] <= STEP_REL_L2, (step, r["rel"])
        # the argmax decision, in the kernel's own float32 precision, is exact
        assert np.array_equal(r["g_next"], oracle.argmax_f32(r["g_logits"]))
        assert rel_l2(r["g_logits"], r["o_logits"]) <= STEP_REL_L2
        # the LM head element by element on the GPU's final hidden rows, and
        # the token against the oracle's argmax
        check_lm_head(r["g_fh"], s.model["lm_head"], r["g_logits"], r["g_next"])
        agree.append(np.mean(r["g_next"] == r["o_next"]))
        tokens = r["o_next"]            # teacher forcing with the oracle's tokens
    assert np.mean(agree) >= 0.8
    # the caches hold every layer's rotated K and V of every step: with both
    # sides fed the same tokens they are identical
    for l in range(cfg["num_layers"]):
        assert np.array_equal(to_host(s.gkc[l]), s.kc[l]), l
        assert np.array_equal(to_host(s.gvc[l]), s.vc[l]), l
    assert a8w8.read_device_errors() == 0


def test_graph_replay_matches_direct_call(a8w8):
    import torch
    cfg = dict(synth.TINY, num_layers=2, vocab=1000)
    B = 2
    s = Session(a8w8, cfg, B, max_seq=64, seed=400)
    g = a8w8.StepGraph(s.gm, cfg, B, s.max_blocks, s.gkc, s.gvc, s.rope, s.ws,
                       logits=s.logits, final_hidden=s.fh)
    tok, slots, ctx = s.inputs([5, 7])
    saved = [c.clone() for c in s.gkc + s.gvc]

    def restore():
        for c, sv in zip(s.gkc + s.gvc, saved):
            c.copy_(sv)

    a8w8.a8w8_decode_step(s.gm, cfg, to_dev(tok), to_dev(slots), to_dev(s.bt), to_dev(ctx), s.gkc,
                          s.gvc, s.rope, s.ws, s.next, logits=s.logits, final_hidden=s.fh)
    d_next, d_fh, d_logits = to_host(s.next), to_host(s.fh), to_host(s.logits)
    d_caches = [to_host(c) for c in s.gkc + s.gvc]
    # host-buffer entry point: copies in, replays, copies out, synchronises
    restore()
    h_next = torch.empty(B, dtype=torch.int32).pin_memory()
    g.run_host(torch.from_numpy(tok).pin_memory(), torch.from_numpy(slots).pin_memory(),
               torch.from_numpy(s.bt.copy()).pin_memory(), torch.from_numpy(ctx).pin_memory(),
               h_next)
    assert np.array_equal(h_next.numpy(), d_next)
    assert np.array_equal(to_host(s.fh), d_fh)
    assert np.array_equal(to_host(s.logits), d_logits)
    assert all(np.array_equal(to_host(c), d) for c, d in zip(s.gkc + s.gvc, d_caches))
    # replay from device-resident inputs
    restore()
    g.set_inputs(to_dev(tok), to_dev(slots), to_dev(s.bt), to_dev(ctx))
    g.launch()
    torch.cuda.synchronize()
    assert np.array_equal(to_host(g.next_tokens), d_next)
    g.close()


def test_device_loop_matches_host_loop(a8w8):
    """Replaying the device-loop graph n times equals n steps fed from the host."""
    import torch
    cfg = dict(synth.TINY, num_layers=2, vocab=777)
    B, n = 3, 12
    s = Session(a8w8, cfg, B, max_seq=48, seed=450)
    saved = [c.clone() for c in s.gkc + s.gvc]
    tok0, slots0, ctx0 = s.inputs(synth.prompt_ids(451, B, cfg["vocab"]))
    # host loop through the direct entry point
    tok, slots, ctx = tok0, slots0, ctx0
    host_tokens = []
    for _ in range(n):
        a8w8.a8w8_decode_step(s.gm, cfg, to_dev(tok), to_dev(slots), to_dev(s.bt), to_dev(ctx),
                              s.gkc, s.gvc, s.rope, s.ws, s.next)
        nxt = to_host(s.next)
        host_tokens.append(nxt)
        tok = nxt
        ctx = ctx + 1
        slots = synth.slots_for(s.bt, ctx - 1, s.page)
    host_caches = [to_host(c) for c in s.gkc + s.gvc]
    for c, sv in zip(s.gkc + s.gvc, saved):
        c.copy_(sv)
    g = a8w8.StepGraph(s.gm, cfg, B, s.max_blocks, s.gkc, s.gvc, s.rope, s.ws, device_loop=True)
    g.set_inputs(to_dev(tok0), to_dev(slots0), to_dev(s.bt), to_dev(ctx0))
    dev_tokens = []
    for _ in range(n):
        g.launch()
        dev_tokens.append(to_host(g.next_tokens))
    assert np.array_equal(np.array(dev_tokens), np.array(host_tokens))
    assert all(np.array_equal(to_host(c), h) for c, h in zip(s.gkc + s.gvc, host_caches))
    assert np.array_equal(to_host(g.ctx_lens), ctx0 + n)
    g.close()


def test_step_bad_token_id_is_flagged(a8w8):
    cfg = dict(synth.TINY, num_layers=1, vocab=100)
    s = Session(a8w8, cfg, 2, max_seq=16, seed=500)
    tok, slots, ctx = s.inputs([3, 100])
    a8w8.read_device_errors()
    a8w8.a8w8_decode_step(s.gm, cfg, to_dev(tok), to_dev(slots), to_dev(s.bt), to_dev(ctx), s.gkc,
                          s.gvc, s.rope, s.ws, s.next)
    assert a8w8.read_device_errors() & a8w8.DEVERR_TOKEN


# Shapes the persistent single-kernel step accepts (head_dim 128, hidden and
# Hq * head_dim multiples of 512, intermediate a multiple of 1024), small enough
# for the oracle.
SMALL_PERSISTENT = dict(synth.TINY, hidden=512, num_q_heads=4, num_kv_heads=2, head_dim=128,
                        intermediate=1024, num_layers=2, vocab=1000, page_size=16)


def _run_steps(a8w8, cfg, B, max_seq, seed, n_steps, flags):
    """n teacher-free steps through the direct entry point; returns per-step
    (next tokens, final hidden, logits) and the caches."""
    c = dict(cfg, flags=flags)
    s = Session(a8w8, c, B, max_seq=max_seq, seed=seed)
    tok, slots, ctx = s.inputs(synth.prompt_ids(seed + 7, B, cfg["vocab"]))
    out = []
    for _ in range(n_steps):
        a8w8.a8w8_decode_step(s.gm, c, to_dev(tok), to_dev(slots), to_dev(s.bt), to_dev(ctx),
                              s.gkc, s.gvc, s.rope, s.ws, s.next, logits=s.logits,
                              final_hidden=s.fh)
        out.append((to_host(s.next), to_host(s.fh), to_host(s.logits)))
        tok = to_host(s.next)
        ctx = ctx + 1
        slots = synth.slots_for(s.bt, ctx - 1, s.page)
    return out, [to_host(x) for x in s.gkc + s.gvc]


@pytest.mark.parametrize("B,max_seq", [(1, 40), (2, 300), (4, 40)])
def test_persistent_step_equals_separate_kernels(a8w8, B, max_seq):
    # max_seq 300 gives 19 pages of 16 tokens: three 128-token KV chunks and a
    # combine pass inside the persistent kernel
    a, ca = _run_steps(a8w8, SMALL_PERSISTENT, B, max_seq, 600 + B, 6, a8w8.FLAG_PERSISTENT_STEP)
    b, cb = _run_steps(a8w8, SMALL_PERSISTENT, B, max_seq, 600 + B, 6, 0)
    for (n1, h1, l1), (n2, h2, l2) in zip(a, b):
        assert np.array_equal(n1, n2)
        assert np.array_equal(h1, h2)
        assert np.array_equal(l1, l2)
    for x, y in zip(ca, cb):
        assert np.array_equal(x, y)
    assert a8w8.read_device_errors() == 0


@pytest.mark.parametrize("B", [1, 4])
def test_persistent_step_teacher_forced_vs_oracle(a8w8, B):
    s = Session(a8w8, dict(SMALL_PERSISTENT, flags=a8w8.FLAG_PERSISTENT_STEP), B, max_seq=48,
                seed=700 + B)
    tokens = synth.prompt_ids(701 + B, B, SMALL_PERSISTENT["vocab"])
    for step in range(12):
        r = s.step_both(tokens)
        assert r["rel"] <= STEP_REL_L2, (step, r["rel"])
        assert np.array_equal(r["g_next"], oracle.argmax_f32(r["g_logits"]))
        assert rel_l2(r["g_logits"], r["o_logits"]) <= STEP_REL_L2
        check_lm_head(r["g_fh"], s.model["lm_head"], r["g_logits"], r["g_next"])
        tokens = r["o_next"]
    assert a8w8.read_device_errors() == 0


def test_persistent_device_loop(a8w8):
    cfg = dict(SMALL_PERSISTENT, flags=a8w8.FLAG_PERSISTENT_STEP)
    B, n = 2, 10
    s = Session(a8w8, cfg, B, max_seq=32, seed=800)
    saved = [c.clone() for c in s.gkc + s.gvc]
    tok0, slots0, ctx0 = s.inputs(synth.prompt_ids(801, B, cfg["vocab"]))
    ref = []
    tok, slots, ctx = tok0, slots0, ctx0
    for _ in range(n):
        a8w8.a8w8_decode_step(s.gm, cfg, to_dev(tok), to_dev(slots), to_dev(s.bt), to_dev(ctx),
                              s.gkc, s.gvc, s.rope, s.ws, s.next)
        ref.append(to_host(s.next))
        tok, ctx = ref[-1], ctx + 1
        slots = synth.slots_for(s.bt, ctx - 1, s.page)
    for c, sv in zip(s.gkc + s.gvc, saved):
        c.copy_(sv)
    g = a8w8.StepGraph(s.gm, cfg, B, s.max_blocks, s.gkc, s.gvc, s.rope, s.ws, device_loop=True)
    g.set_inputs(to_dev(tok0), to_dev(slots0), to_dev(s.bt), to_dev(ctx0))
    got = []
    for _ in range(n):
        g.launch()
        got.append(to_host(g.next_tokens))
    assert np.array_equal(np.array(got), np.array(ref))
    g.close()




def test_qwen3_14b_lm_head_full_vocab_vs_oracle(a8w8):
    """The final norm, the 151936-row BF16 LM head and the argmax at full
    size (one Qwen3-14B-shaped layer in front, batch 2), element by element
    on the GPU's own final hidden rows."""
    import torch
    cfg = dict(synth.QWEN3_14B, num_layers=1)
    dev = torch.device("cuda")
    model = synth.t_model_weights(cfg, 77, dev)
    B, page, Hkv, D = 2, cfg["page_size"], cfg["num_kv_heads"], cfg["head_dim"]
    kc = [torch.zeros((2 * page, Hkv, D), dtype=torch.bfloat16, device=dev)]
    vc = [torch.zeros_like(kc[0])]
    rope = a8w8.a8w8_rope_table(page, D, cfg["rope_theta"])
    ws = a8w8.alloc_workspace(cfg, B, 1)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    logits = torch.empty((B, cfg["vocab"]), dtype=torch.float32, device=dev)
    fh = torch.empty((B, cfg["hidden"]), dtype=torch.bfloat16, device=dev)
    bt = np.array([[0], [1]], np.int32)
    tok = synth.prompt_ids(78, B, cfg["vocab"])
    ctx = np.array([1, 1], np.int32)
    slots = synth.slots_for(bt, ctx - 1, page)
    a8w8.a8w8_decode_step(model, cfg, to_dev(tok), to_dev(slots), to_dev(bt), to_dev(ctx), kc, vc,
                          rope, ws, nxt, logits=logits, final_hidden=fh)
    torch.cuda.synchronize()
    W = model["lm_head"].detach().cpu().view(torch.int16).numpy().view(np.uint16)
    worst, ties = check_lm_head(to_host(fh), W, to_host(logits), to_host(nxt))
    print("LM head: worst |diff| / bound", worst, "near ties", ties)
    assert a8w8.read_device_errors() == 0


@pytest.mark.parametrize("T,top_p", [(0.8, 0.9), (1.3, 1.0), (0.0, 1.0)])
def test_sampled_device_loop_graph(a8w8, T, top_p):
    """Sampling inside the replayed step graph: replay i draws exactly what
    a8w8_sample draws from that replay's logits at step s0 + i (the same
    kernels), which agrees with the oracle's sampling rule; the drawn tokens
    are fed back as the next step's tokens and the step counter advances by
    one per replay; temperature 0 gives the argmax of the logits."""
    import torch
    cfg = dict(synth.TINY, num_layers=2, vocab=777)
    B, n, seed, s0 = 3, 8, 0xABCDEF12345, 5
    s = Session(a8w8, cfg, B, max_seq=48, seed=460)
    tok0, slots0, ctx0 = s.inputs(synth.prompt_ids(461, B, cfg["vocab"]))
    g = a8w8.StepGraph(s.gm, cfg, B, s.max_blocks, s.gkc, s.gvc, s.rope, s.ws, logits=s.logits,
                       device_loop=True,
                       sampling=dict(temperature=T, top_p=top_p, seed=seed, step=s0))
    g.set_inputs(to_dev(tok0), to_dev(slots0), to_dev(s.bt), to_dev(ctx0))
    agree = 0
    for i in range(n):
        g.launch()
        torch.cuda.synchronize()
        got = to_host(g.next_tokens)
        lg = to_host(s.logits)
        same = to_host(a8w8.a8w8_sample(s.logits, T, top_p, seed=seed, step=s0 + i))
        assert np.array_equal(got, same), (i, got, same)
        if T > 0:
            agree += int((got == sampling.sample_rows(lg, T, top_p, seed, s0 + i)).sum())
        else:
            assert np.array_equal(got, np.argmax(lg, axis=1))
        assert np.array_equal(to_host(g.token_ids), got)        # fed back on the device
    if T > 0:
        # float32 Gumbel keys on the device, float64 in the oracle (as for a8w8_sample)
        assert agree >= n * B - 1, (agree, n * B)
    assert int(to_host(g.step_counter)[0]) == s0 + n
    assert np.array_equal(to_host(g.ctx_lens), ctx0 + n)
    g.close()

