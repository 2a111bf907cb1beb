"""GPU parity of the decode step (embedding, layers, final norm, LM head,
greedy argmax) against the oracle, plus the replayable graph and the
host-buffer entry point."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import STEP_REL_L2, bf16_to_f64, rel_l2, to_dev, to_host

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
                    g_logits=g_logits, o_logits=o_logits)


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
        agree.append(np.mean(r["g_next"] == r["o_next"]))
        tokens = r["o_next"]            # teacher forcing with the oracle's tokens
    assert np.mean(agree) >= 0.8
    # caches stay close to the oracle's (they hold the per-layer rotated K and V)
    for l in range(cfg["num_layers"]):
        assert rel_l2(bf16_to_f64(to_host(s.gkc[l])), bf16_to_f64(s.kc[l])) <= 2e-2
        assert rel_l2(bf16_to_f64(to_host(s.gvc[l])), bf16_to_f64(s.vc[l])) <= 2e-2
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
