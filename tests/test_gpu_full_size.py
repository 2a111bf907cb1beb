"""The benchmarked 40-layer Qwen3-14B-shaped decode steps at full size against
the oracle: batch 1 with the 151936-row LM head (the headline workload) and
batch 16 with contexts drawn from [64, 4096] over shuffled pages.

Weights are drawn on the device as in the benchmark; the oracle reads host
copies. Both sides start each compared step from the same KV caches (the
GPU's, copied to the host): a step is 40 quantised layers deep, and
differences carried in the caches from earlier steps would compound with the
step's own. The step runs through the same replayable graph the benchmark
times.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import STEP_REL_L2, bf16_to_f64, check_lm_head, rel_l2, to_dev, to_host

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def a8w8():
    import w8a8_quantized_decode_gb300 as m
    m.build()
    return m


def _host(t):
    import torch
    t = t.detach().cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


@pytest.fixture(scope="module")
def qwen3(a8w8):
    """The 40-layer model on the device and its host copy (drawn once)."""
    import torch
    cfg = dict(synth.QWEN3_14B)
    model = synth.t_model_weights(cfg, 2026, torch.device("cuda"))
    hm = dict(embed=_host(model["embed"]), final_norm_w=_host(model["final_norm_w"]),
              lm_head=_host(model["lm_head"]),
              layers=[{k: _host(v) for k, v in l.items()} for l in model["layers"]])
    return cfg, model, hm


class FullStep:
    """The step graph over device caches, with host mirrors for the oracle."""

    def __init__(self, a8w8, cfg, model, B, bt, nblk, gen_seed=None):
        import torch
        self.a8w8, self.cfg, self.B, self.bt = a8w8, cfg, B, bt
        page, Hkv, D, L = cfg["page_size"], cfg["num_kv_heads"], cfg["head_dim"], cfg["num_layers"]
        dev = torch.device("cuda")
        shape = (nblk * page, Hkv, D)
        if gen_seed is None:
            self.kc = [torch.zeros(shape, dtype=torch.bfloat16, device=dev) for _ in range(L)]
            self.vc = [torch.zeros(shape, dtype=torch.bfloat16, device=dev) for _ in range(L)]
        else:
            g = torch.Generator(device=dev)
            g.manual_seed(gen_seed)
            self.kc, self.vc = [], []
            for _ in range(L):
                self.kc.append(torch.randn(shape, generator=g, device=dev).to(torch.bfloat16))
                self.vc.append(torch.randn(shape, generator=g, device=dev).to(torch.bfloat16))
        max_blocks = bt.shape[1]
        self.rope = a8w8.a8w8_rope_table(max_blocks * page, D, cfg["rope_theta"])
        self.ws = a8w8.alloc_workspace(cfg, B, max_blocks)
        self.fh = torch.empty((B, cfg["hidden"]), dtype=torch.bfloat16, device=dev)
        self.logits = torch.empty((B, cfg["vocab"]), dtype=torch.float32, device=dev)
        self.g = a8w8.StepGraph(model, cfg, B, max_blocks, self.kc, self.vc, self.rope, self.ws,
                                logits=self.logits, final_hidden=self.fh)

    def run(self, tok, ctx):
        import torch
        slots = synth.slots_for(self.bt, ctx - 1, self.cfg["page_size"])
        self.g.set_inputs(to_dev(tok), to_dev(slots), to_dev(self.bt), to_dev(ctx))
        self.g.launch()
        torch.cuda.synchronize()
        return slots, to_host(self.g.next_tokens)

    def compare(self, hm, tok, ctx):
        """One step on both sides from the GPU's current caches."""
        okc = [to_host(c) for c in self.kc]
        ovc = [to_host(c) for c in self.vc]
        slots, g_next = self.run(tok, ctx)
        o_next, o_fh, o_logits, rc = oracle.decode_step(hm, self.cfg, tok, slots, self.bt, ctx,
                                                        okc, ovc, want_logits=True)
        assert rc == 0
        g_fh = to_host(self.fh)
        rel = rel_l2(bf16_to_f64(g_fh), bf16_to_f64(o_fh))
        same = float((g_fh == o_fh).mean())
        assert rel <= STEP_REL_L2, rel
        g_logits = to_host(self.logits)
        assert rel_l2(g_logits, o_logits) <= STEP_REL_L2
        # the LM head element by element on the GPU's own final hidden rows
        worst, ties = check_lm_head(g_fh, hm["lm_head"], g_logits, g_next)
        # the caches the step wrote (every layer's K and V at the new slots)
        kv_same = min(float((to_host(c) == o).mean()) for c, o in zip(self.kc + self.vc, okc + ovc))
        return dict(rel=rel, identical=same, lm_worst=worst, near_ties=ties, kv_identical=kv_same,
                    tokens_equal=float((g_next == o_next).mean())), o_next, g_next

    def close(self):
        self.g.close()


def test_qwen3_14b_40_layer_step_b1_vs_oracle(a8w8, qwen3):
    """The headline workload: batch 1, a 16-token prompt decoded through the
    step graph, then steps compared with the oracle at contexts 17, 18 and
    64 (the benchmark times contexts 17 to 64)."""
    cfg, model, hm = qwen3
    bt = np.array([[0, 1]], np.int32)
    s = FullStep(a8w8, cfg, model, 1, bt, 2)
    tok = synth.prompt_ids(5, 16, cfg["vocab"])
    for i in range(16):                      # the prompt, one token per step
        cur = s.run(tok[i:i + 1], np.array([i + 1], np.int32))[1]
    reports = []
    for ctx in range(17, 65):
        c = np.array([ctx], np.int32)
        if ctx in (17, 18, 64):
            rep, cur, _ = s.compare(hm, cur, c)     # teacher forcing: the oracle's token
            reports.append((ctx, rep))
        else:
            cur = s.run(cur, c)[1]
    print("40-layer batch-1 steps:", reports)
    s.close()
    assert a8w8.read_device_errors() == 0


def test_qwen3_14b_40_layer_step_b16_vs_oracle(a8w8, qwen3):
    """Batched paged decode at full size: batch 16, contexts uniform in
    [64, 4096], block tables from a shuffled permutation of the physical
    pages, N(0, 1) context K/V, two teacher-forced steps."""
    cfg, model, hm = qwen3
    B, page = 16, cfg["page_size"]
    ctx0 = synth.batched_ctx_lens(9020, B)
    bt, nblk = synth.paged_layout(9021, ctx0, page, extra_tokens=2)
    s = FullStep(a8w8, cfg, model, B, bt, nblk, gen_seed=9022)
    tok = synth.prompt_ids(9023, B, cfg["vocab"])
    reports = []
    for step in range(2):
        rep, o_next, _ = s.compare(hm, tok, (ctx0 + step).astype(np.int32))
        reports.append(rep)
        tok = o_next
    print("40-layer batch-16 steps (contexts", ctx0.tolist(), "):", reports)
    s.close()
    assert a8w8.read_device_errors() == 0
