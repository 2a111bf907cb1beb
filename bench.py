"""Benchmark of the A8W8 decode step on GB300.

Workload (default): a 40-layer Qwen3-14B-shaped A8W8 decode step with the BF16
LM head and greedy argmax, batch 1. A 16-token seeded prompt is decoded token by
token to fill the paged BF16 KV cache, then W warm-up steps and K timed steps
follow (max_seq_len 256). Weights are random-init (seeded, drawn on the device),
14.8 GB per step, far larger than L2, so no step can hit in L2 for weights.

value    : TPOT (ms/token) of K replays of the captured step graph whose inputs
           stay in HBM (the graph feeds each argmax back as the next token).
e2e      : TPOT through the C ABI with HOST buffers: every step copies its
           inputs from pinned host memory and reads the next token back.
roofline : the Gate/Up projection kernel (54% of the step's bytes), timed live
           with CUDA events over the 40 layers' Gate/Up weights.
cpu_baseline / --impl reference : the CPU oracle, timed on one decode step.

--workload batched16: the batched paged decode step instead (batch 16, contexts
drawn uniformly from [64, 4096], pages of 128 tokens in a seeded shuffled
permutation, synthetic N(0,1) context K/V, each new token written into its
request's last page), K replays of the device-loop step graph (default 32
steps); one JSON line with the step time, tokens/s and the step's HBM bytes.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload decode_b1|batched16]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

PROMPT_LEN = 16
MAX_SEQ = 256
SEED = 2026
WORKLOAD = "qwen3_14b_a8w8_decode_step_b1"
METRIC = "A8W8 decode TPOT (ms/token, 40 layers, bs=1)"

# DRAM bytes (read + write) per launch of the fused post-attention norm +
# Gate/Up + SwiGLU kernel the step runs (gemv_stream_kernel<1, 2, 1, 1, 6, 2>),
# from an ncu capture of the kernel as it is now built (the batch-1 layer
# capture: 178,481,664 read + 2,923,264 written); None while no capture of the
# current kernel exists.
GATE_UP_NCU_TRAFFIC_BYTES = 181404928


def step_bytes(cfg, ctx_lens) -> dict:
    """Algorithmic bytes of one decode step (weights, norms, KV read + write)."""
    H, V, L = cfg["hidden"], cfg["vocab"], cfg["num_layers"]
    Hkv, D = cfg["num_kv_heads"], cfg["head_dim"]
    layer = synth.layer_weight_bytes(cfg)
    kv_row = 2 * Hkv * D * 2            # K and V of one token, one layer
    kv = sum(int(c) for c in ctx_lens) * kv_row * L   # read (the new token is written once)
    head = V * H * 2 + H * 2
    return {"layers": layer * L, "lm_head": head, "kv": kv, "total": layer * L + head + kv}


def gate_up_bytes(cfg, B: int = 1) -> int:
    """Algorithmic bytes of one launch of the fused a11-a12 kernel: the Gate/Up
    weights and scales, the post-attention norm weight, the BF16 input rows
    and the SwiGLU output rows."""
    H, I = cfg["hidden"], cfg["intermediate"]
    return 2 * I * H + 2 * I * 4 + H * 2 + B * H * 2 + B * I * 2


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "20"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def max_over_ranks(value: float, device=None) -> float:
    """The maximum of a per-rank timing over all ranks (the job ends with its
    slowest replica); the value itself when the run is not distributed. NCCL
    reduces a tensor on the rank's GPU, gloo one on the CPU."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, ms_max: float, world: int) -> float:
    """Whole-job throughput per second: every rank (a replica) processes the
    same units, and the job takes the slowest rank's time."""
    return units_per_rank * world * 1000.0 / ms_max


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def build_model(cfg, device):
    import torch
    m = synth.t_model_weights(cfg, SEED, device)
    torch.cuda.synchronize()
    return m


def host_model(model) -> dict:
    """Copy a device model to numpy (BF16 as uint16) for the oracle."""
    import torch

    def h(t):
        t = t.detach().cpu()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()
    return dict(embed=h(model["embed"]), final_norm_w=h(model["final_norm_w"]),
                lm_head=h(model["lm_head"]),
                layers=[{k: h(v) for k, v in l.items()} for l in model["layers"]])


def host_cpu(cpuinfo: str = "/proc/cpuinfo") -> dict:
    """The host CPU's model and logical core count, for the oracle timings
    (never raises: unknown fields read "unknown")."""
    model = None
    arm = {}
    try:
        with open(cpuinfo) as f:
            for ln in f:
                if ":" not in ln:
                    continue
                key, val = (x.strip() for x in ln.split(":", 1))
                key = key.lower()
                if key == "model name" and not model:
                    model = val
                elif key in ("cpu implementer", "cpu part") and key not in arm:
                    arm[key] = val
    except (OSError, UnicodeDecodeError):
        pass
    if not model and arm:
        model = (f"implementer {arm.get('cpu implementer', '?')} "
                 f"part {arm.get('cpu part', '?')}")
    import platform
    return {"model": model or platform.processor() or "unknown",
            "arch": platform.machine() or "unknown", "nproc": os.cpu_count()}


def time_oracle_steps(hm, cfg, n_steps: int, budget_s: float):
    """Oracle decode steps (batch 1) from a prompt of PROMPT_LEN tokens; returns
    (seconds per step list, threads)."""
    import oracle
    page = cfg["page_size"]
    max_blocks = MAX_SEQ // page
    bt = np.arange(max_blocks, dtype=np.int32)[None, :]
    Hkv, D = cfg["num_kv_heads"], cfg["head_dim"]
    L = cfg["num_layers"]
    kc = [np.zeros((max_blocks * page, Hkv, D), np.uint16) for _ in range(L)]
    vc = [np.zeros((max_blocks * page, Hkv, D), np.uint16) for _ in range(L)]
    tok = synth.prompt_ids(SEED + 5, 1, cfg["vocab"])
    times = []
    t_start = time.perf_counter()
    for s in range(n_steps):
        ctx = np.array([PROMPT_LEN + s + 1], np.int32)
        slots = synth.slots_for(bt, ctx - 1, page)
        t0 = time.perf_counter()
        nxt, _, _, rc = oracle.decode_step(hm, cfg, tok, slots, bt, ctx, kc, vc)
        times.append(time.perf_counter() - t0)
        tok = nxt
        if time.perf_counter() - t_start > budget_s:
            break
    return times, oracle.num_threads()


def run_reference(args, cfg):
    """The oracle as the reference arm (rank 0 only)."""
    import torch
    rank, world, local = dist_env()
    if rank != 0:
        return
    device = torch.device(f"cuda:{local}") if torch.cuda.is_available() else None
    if device is not None:
        torch.cuda.set_device(device)
        model = build_model(cfg, device)
        hm = host_model(model)
        del model
        torch.cuda.empty_cache()
    else:
        hm = synth.model_weights_host(cfg, SEED)
    import oracle
    oracle.build()
    n = args.warmup + args.steps
    times, threads = time_oracle_steps(hm, cfg, n, budget_s=240.0)
    timed = times[args.warmup:] if len(times) > args.warmup else times
    tpot = 1000.0 * sum(timed) / len(timed)
    line = {
        "impl": "reference", "metric": METRIC, "value": tpot, "unit": "ms/token",
        "n_gpus": args.gpus, "steps": len(timed), "warmup": min(args.warmup, len(times)),
        "ms_per_step": tpot, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8/int32/f32/f64", "data": "synthetic (seeded random-init weights)",
        "config": {"workload": WORKLOAD, "batch": 1, "prompt_len": PROMPT_LEN,
                   "max_seq_len": MAX_SEQ, "layers": cfg["num_layers"]},
        "cpu_baseline": {"value": tpot, "unit": "ms/token", "cores": threads, "kind": "oracle",
                         "host": host_cpu(),
                         "sample": f"{len(timed)} oracle decode steps (40 layers + LM head, "
                                   f"batch 1, context {PROMPT_LEN + 1}..)"},
        "e2e": {"value": tpot, "unit": "ms/token", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, cfg):
    import torch
    import w8a8_quantized_decode_gb300 as a8w8

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    a8w8.build()
    B = 1
    page = cfg["page_size"]
    max_blocks = MAX_SEQ // page
    n_total = PROMPT_LEN + args.warmup + args.steps
    if n_total > MAX_SEQ:
        raise SystemExit(f"prompt + warmup + steps = {n_total} exceeds max_seq_len {MAX_SEQ}")

    model = build_model(cfg, device)
    Hkv, D, L = cfg["num_kv_heads"], cfg["head_dim"], cfg["num_layers"]
    nblk = max_blocks + 1
    perm = np.random.default_rng(SEED + 1).permutation(nblk).astype(np.int32)
    bt = perm[:max_blocks][None, :]
    kc = [torch.zeros((nblk * page, Hkv, D), dtype=torch.bfloat16, device=device) for _ in range(L)]
    vc = [torch.zeros((nblk * page, Hkv, D), dtype=torch.bfloat16, device=device) for _ in range(L)]
    rope = a8w8.a8w8_rope_table(MAX_SEQ, D, cfg["rope_theta"], device=device)
    ws = a8w8.alloc_workspace(cfg, B, max_blocks, device=device)
    stream = torch.cuda.Stream(device)

    # device-resident decode loop: the graph feeds each argmax back on the device
    with torch.cuda.stream(stream):
        g = a8w8.StepGraph(model, cfg, B, max_blocks, kc, vc, rope, ws, device_loop=True,
                           stream=stream)
        prompt = synth.prompt_ids(SEED + 5, PROMPT_LEN, cfg["vocab"])
        # prompt: one step per token, the next prompt token overriding the argmax
        g.block_table.copy_(torch.from_numpy(bt))
        for i in range(PROMPT_LEN):
            ctx = np.array([i + 1], np.int32)
            g.token_ids.copy_(torch.from_numpy(prompt[i:i + 1]))
            g.ctx_lens.copy_(torch.from_numpy(ctx))
            g.slot_mapping.copy_(torch.from_numpy(synth.slots_for(bt, ctx - 1, page)))
            g.launch(stream)
        for _ in range(args.warmup):
            g.launch(stream)
        stream.synchronize()
        gpu_uuid = None
        try:
            gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            pass
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        with ClockSampler(gpu_uuid) as clocks:
            ev0.record(stream)
            for _ in range(args.steps):
                g.launch(stream)
            ev1.record(stream)
            ev1.synchronize()
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1)
        ctx_timed = [PROMPT_LEN + args.warmup + i + 1 for i in range(args.steps)]
        ms = max_over_ranks(ms, device)
        tpot = ms / args.steps
        errs = a8w8.read_device_errors(stream)

        # e2e: host buffers through the C ABI, inputs H2D + next token D2H every step
        e2e_graph = a8w8.StepGraph(model, cfg, B, max_blocks, kc, vc, rope, ws, device_loop=False,
                                   stream=stream)
        h_tok = torch.zeros(B, dtype=torch.int32).pin_memory()
        h_slot = torch.zeros(B, dtype=torch.int32).pin_memory()
        h_bt = torch.from_numpy(bt.copy()).pin_memory()
        h_ctx = torch.zeros(B, dtype=torch.int32).pin_memory()
        h_next = torch.zeros(B, dtype=torch.int32).pin_memory()
        # numpy views of the pinned buffers: the per-step host updates are
        # plain stores into the memory the copies read
        n_tok, n_slot, n_ctx, n_next = (t.numpy() for t in (h_tok, h_slot, h_ctx, h_next))
        n_tok[0] = int(prompt[-1])

        def e2e_step(pos):
            n_ctx[0] = pos + 1
            n_slot[0] = int(bt[0, pos // page]) * page + pos % page
            e2e_graph.run_host(h_tok, h_slot, h_bt, h_ctx, h_next, stream=stream)
            n_tok[0] = n_next[0]

        for i in range(args.warmup):
            e2e_step(PROMPT_LEN + i)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(args.steps):
            e2e_step(PROMPT_LEN + args.warmup + i)
        e2e_ms = (time.perf_counter() - t0) * 1000.0 / args.steps
        h2d = (B + B + B * max_blocks + B) * 4
        d2h = B * 4
        e2e_graph.close()

        # roofline of the dominant kernel, the one the step runs for a11-a12:
        # post-attention RMSNorm and quantisation of the BF16 row in the
        # prologue, Gate/Up + SwiGLU, over the 40 layers' weights (13.2 GB >
        # L2), its 40 launches replayed as one CUDA graph on `stream`
        gu_bytes = gate_up_bytes(cfg, B)
        xrow = synth.t_bf16_normal(SEED + 40, (B, cfg["hidden"]), device, std=30.0)
        act = torch.empty((B, cfg["intermediate"]), dtype=torch.bfloat16, device=device)

        def gate_up_all():
            for l in range(L):
                lw = model["layers"][l]
                a8w8.a8w8_rmsnorm_gate_up_swiglu(xrow, lw["post_norm_w"], cfg["rms_eps"],
                                                 lw["w_gate_up"], lw["s_gate_up"], out=act,
                                                 stream=stream)
        gate_up_all()
        stream.synchronize()
        gg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gg, stream=stream):
            gate_up_all()
        for _ in range(2):
            gg.replay()
        reps = 3
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        stream.synchronize()
        e0.record(stream)
        for _ in range(reps):
            gg.replay()
        e1.record(stream)
        e1.synchronize()
        gu_ms = e0.elapsed_time(e1) / (reps * L)
        del gg

    peaks = measured_peaks()
    sb = step_bytes(cfg, ctx_timed)
    per_step_bytes = sb["layers"] + sb["lm_head"] + sb["kv"] / args.steps
    achieved = gu_bytes / (gu_ms * 1e-3) / 1e9
    n_launch = 1 + L * 5 + 1 + 1     # embed, 5 per layer, LM head, device-loop advance
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(model, cfg)
    if rank == 0:
        line = {
            "metric": METRIC, "value": tpot, "unit": "ms/token", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tpot,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8 x int8 -> int32, f32 dequant, bf16 activations",
            "data": "synthetic (seeded random-init weights drawn on the device)",
            "config": {"workload": WORKLOAD, "batch": 1, "layers": L, "hidden": cfg["hidden"],
                       "intermediate": cfg["intermediate"], "vocab": cfg["vocab"],
                       "prompt_len": PROMPT_LEN, "max_seq_len": MAX_SEQ, "page_size": page,
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (14.8 GB of weights per step)"},
            "tokens_per_s": job_rate(1, tpot, world),
            "step_bytes": per_step_bytes,
            "step_hbm_gbs": per_step_bytes / (tpot * 1e-3) / 1e9,
            "step_frac_of_peak": per_step_bytes / (tpot * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "layers_frac": sb["layers"] / (tpot * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "e2e": {"value": e2e_ms, "unit": "ms/token", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": n_launch * args.steps,
            "roofline": {"bound": "hbm",
                         "kernel": "post-attention RMSNorm + quant + Gate/Up + SwiGLU "
                                   "(gemv_stream_kernel<1, PRO_NORM_QUANT, EPI_SWIGLU, 1>)",
                         "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"],
                         "traffic": GATE_UP_NCU_TRAFFIC_BYTES,
                         "bytes_per_launch": gu_bytes, "ms_per_launch": gu_ms,
                         "peak_source": peaks["source"] + " (HBM copy GB/s, MEASURED_PEAKS.json)"},
            "clocks": clocks.summary(),
            "device_errors": errs,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


SAMPLED_T, SAMPLED_TOP_P = 0.8, 0.95


def run_sampled(args, cfg):
    """The headline workload (40 layers, batch 1, 16-token prompt, max_seq_len
    256) decoded with temperature / top-p sampling inside the replayed
    device-loop graph (a8w8_step_graph_create_sampled): TPOT with the sampler
    over the full vocabulary in every step."""
    import torch
    import w8a8_quantized_decode_gb300 as a8w8

    device = torch.device("cuda:0")
    torch.cuda.set_device(device)
    a8w8.build()
    B, page = 1, cfg["page_size"]
    max_blocks = MAX_SEQ // page
    if PROMPT_LEN + args.warmup + args.steps > MAX_SEQ:
        raise SystemExit("prompt + warmup + steps exceeds max_seq_len")
    model = build_model(cfg, device)
    Hkv, D, L = cfg["num_kv_heads"], cfg["head_dim"], cfg["num_layers"]
    nblk = max_blocks + 1
    bt = np.random.default_rng(SEED + 1).permutation(nblk).astype(np.int32)[:max_blocks][None, :]
    kc = [torch.zeros((nblk * page, Hkv, D), dtype=torch.bfloat16, device=device) for _ in range(L)]
    vc = [torch.zeros((nblk * page, Hkv, D), dtype=torch.bfloat16, device=device) for _ in range(L)]
    rope = a8w8.a8w8_rope_table(MAX_SEQ, D, cfg["rope_theta"], device=device)
    ws = a8w8.alloc_workspace(cfg, B, max_blocks, device=device)
    logits = torch.empty((B, cfg["vocab"]), dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        g = a8w8.StepGraph(model, cfg, B, max_blocks, kc, vc, rope, ws, logits=logits,
                           device_loop=True, stream=stream,
                           sampling=dict(temperature=SAMPLED_T, top_p=SAMPLED_TOP_P, seed=SEED,
                                         step=0))
        prompt = synth.prompt_ids(SEED + 5, PROMPT_LEN, cfg["vocab"])
        g.block_table.copy_(torch.from_numpy(bt))
        for i in range(PROMPT_LEN):
            ctx = np.array([i + 1], np.int32)
            g.token_ids.copy_(torch.from_numpy(prompt[i:i + 1]))
            g.ctx_lens.copy_(torch.from_numpy(ctx))
            g.slot_mapping.copy_(torch.from_numpy(synth.slots_for(bt, ctx - 1, page)))
            g.launch(stream)
        for _ in range(args.warmup):
            g.launch(stream)
        stream.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        with ClockSampler(None) as clocks:
            ev0.record(stream)
            for _ in range(args.steps):
                g.launch(stream)
            ev1.record(stream)
            ev1.synchronize()
        tpot = ev0.elapsed_time(ev1) / args.steps
        errs = a8w8.read_device_errors(stream)
        g.close()
    print(json.dumps({
        "metric": "A8W8 decode TPOT with in-graph sampling (ms/token, 40 layers, bs=1)",
        "value": tpot, "unit": "ms/token", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "higher_is_better": False, "vs_baseline": None,
        "dtype": "int8 x int8 -> int32, f32 dequant, bf16 activations; two-float sampling masses",
        "data": "synthetic (seeded random-init weights drawn on the device)",
        "config": {"workload": "qwen3_14b_a8w8_decode_step_b1_sampled", "batch": 1, "layers": L,
                   "vocab": cfg["vocab"], "temperature": SAMPLED_T, "top_p": SAMPLED_TOP_P,
                   "prompt_len": PROMPT_LEN, "max_seq_len": MAX_SEQ},
        "tokens_per_s": 1000.0 / tpot, "gpu_launches": None, "clocks": clocks.summary(),
        "device_errors": errs}), flush=True)


BATCHED_B = 16
BATCHED_WORKLOAD = "qwen3_14b_a8w8_batched_decode_b16"
BATCHED_METRIC = "A8W8 batched decode step (ms/step, 40 layers, bs=16, contexts 64..4096)"


def run_batched(args, cfg):
    """Batch-16 paged decode with long mixed contexts (one GPU per rank)."""
    import torch
    import w8a8_quantized_decode_gb300 as a8w8

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    a8w8.build()
    B, page = BATCHED_B, cfg["page_size"]
    Hkv, D, L = cfg["num_kv_heads"], cfg["head_dim"], cfg["num_layers"]
    ctx0 = synth.batched_ctx_lens(SEED + 20, B)
    grow = args.warmup + args.steps
    bt, nblk = synth.paged_layout(SEED + 21, ctx0, page, extra_tokens=grow)
    max_blocks = bt.shape[1]
    model = build_model(cfg, device)
    gen = torch.Generator(device=device)
    gen.manual_seed(SEED + 22)
    kc, vc = [], []
    for _ in range(L):
        kc.append(torch.randn((nblk * page, Hkv, D), generator=gen, device=device).to(torch.bfloat16))
        vc.append(torch.randn((nblk * page, Hkv, D), generator=gen, device=device).to(torch.bfloat16))
    rope = a8w8.a8w8_rope_table(max_blocks * page, D, cfg["rope_theta"], device=device)
    ws = a8w8.alloc_workspace(cfg, B, max_blocks, device=device)
    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        g = a8w8.StepGraph(model, cfg, B, max_blocks, kc, vc, rope, ws, device_loop=True,
                           stream=stream)
        tok = synth.prompt_ids(SEED + 23, B, cfg["vocab"])
        slots = synth.slots_for(bt, ctx0 - 1, page)
        g.set_inputs(torch.from_numpy(tok).to(device), torch.from_numpy(slots).to(device),
                     torch.from_numpy(bt).to(device),
                     torch.from_numpy(ctx0.astype(np.int32)).to(device))
        for _ in range(args.warmup):
            g.launch(stream)
        stream.synchronize()
        gpu_uuid = None
        try:
            gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            pass
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        with ClockSampler(gpu_uuid) as clocks:
            ev0.record(stream)
            for _ in range(args.steps):
                g.launch(stream)
            ev1.record(stream)
            ev1.synchronize()
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1)
        ms = max_over_ranks(ms, device)
        errs = a8w8.read_device_errors(stream)
        g.close()
    per_step = ms / args.steps
    # contexts of the timed steps: ctx0 + warmup + i + 1 tokens, summed over rows
    ctx_sum = sum(int(c) + args.warmup + i for c in ctx0 for i in range(args.steps))
    sb = step_bytes(cfg, [ctx_sum])
    per_step_bytes = sb["layers"] + sb["lm_head"] + sb["kv"] / args.steps
    peaks = measured_peaks()
    # embed; per layer 4 row quantisations + 4 projections + attention; the LM
    # head in tiles of 8 rows; the device-loop advance
    n_launch = 1 + L * 9 + (B + 7) // 8 + 1
    if rank == 0:
        line = {
            "metric": BATCHED_METRIC, "value": per_step, "unit": "ms/step", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8 x int8 -> int32, f32 dequant, bf16 activations",
            "data": "synthetic (seeded random-init weights and N(0,1) context K/V on the device)",
            "config": {"workload": BATCHED_WORKLOAD, "batch": B, "layers": L,
                       "ctx_range": [64, 4096], "mean_ctx_start": float(ctx0.mean()),
                       "page_size": page, "max_blocks": int(max_blocks),
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (14.8 GB of weights + KV per step)"},
            "tokens_per_s": job_rate(B, per_step, world),
            "step_bytes": per_step_bytes,
            "step_hbm_gbs": per_step_bytes / (per_step * 1e-3) / 1e9,
            "step_frac_of_peak": per_step_bytes / (per_step * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "e2e": None,
            "gpu_launches": n_launch * args.steps,
            "clocks": clocks.summary(),
            "device_errors": errs,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_batched_i8kv(args, cfg):
    """The batch-16 step over INT8 KV caches against the same step over BF16
    caches, both at the seeded contexts (64..4096) held fixed: each replay
    decodes the same positions, so both read the same number of cached rows
    (rank 0 only)."""
    import torch
    import w8a8_quantized_decode_gb300 as a8w8

    rank, world, local = dist_env()
    if rank != 0:
        return
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    a8w8.build()
    B, page = BATCHED_B, cfg["page_size"]
    Hkv, D, L = cfg["num_kv_heads"], cfg["head_dim"], cfg["num_layers"]
    ctx0 = synth.batched_ctx_lens(SEED + 20, B)
    bt_np, nblk = synth.paged_layout(SEED + 21, ctx0, page)
    max_blocks = bt_np.shape[1]
    model = build_model(cfg, device)
    gen = torch.Generator(device=device)
    gen.manual_seed(SEED + 22)
    kc, vc, k8, v8, ks, vs = [], [], [], [], [], []
    for l in range(L):
        kc.append(torch.randn((nblk * page, Hkv, D), generator=gen, device=device).to(torch.bfloat16))
        vc.append(torch.randn((nblk * page, Hkv, D), generator=gen, device=device).to(torch.bfloat16))
        c, sc = synth.t_i8_kv_history(SEED + 100 + 4 * l, nblk * page, Hkv, D, device)
        k8.append(c)
        ks.append(sc)
        c, sc = synth.t_i8_kv_history(SEED + 102 + 4 * l, nblk * page, Hkv, D, device)
        v8.append(c)
        vs.append(sc)
    rope = a8w8.a8w8_rope_table(max_blocks * page, D, cfg["rope_theta"], device=device)
    ws = a8w8.alloc_workspace(cfg, B, max_blocks, device=device)
    tok = torch.from_numpy(synth.prompt_ids(SEED + 23, B, cfg["vocab"])).to(device)
    sl = torch.from_numpy(synth.slots_for(bt_np, ctx0 - 1, page)).to(device)
    bt = torch.from_numpy(bt_np).to(device)
    cl = torch.from_numpy(ctx0.astype(np.int32)).to(device)
    nxt = torch.empty(B, dtype=torch.int32, device=device)
    stream = torch.cuda.Stream(device)
    n = max(args.steps, 4)

    def step(int8):
        if int8:
            a8w8.a8w8_decode_step_i8kv(model, cfg, tok, sl, bt, cl, k8, v8, ks, vs, rope, ws, nxt,
                                       stream=stream)
        else:
            a8w8.a8w8_decode_step(model, cfg, tok, sl, bt, cl, kc, vc, rope, ws, nxt, stream=stream)

    gpu_uuid = None
    try:
        gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass
    ms = {}
    clock_runs = {}
    with torch.cuda.stream(stream):
        for int8 in (False, True):
            step(int8)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(n):
                    step(int8)
            for _ in range(args.warmup):
                g.replay()
            stream.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with ClockSampler(gpu_uuid) as clocks:
                e0.record(stream)
                g.replay()
                e1.record(stream)
                e1.synchronize()
            ms[int8] = e0.elapsed_time(e1) / n
            clock_runs["int8_kv" if int8 else "bf16_kv"] = clocks.summary()
            del g
        errs = a8w8.read_device_errors(stream)
    ctx_sum = int(ctx0.sum())
    sb = step_bytes(cfg, [ctx_sum])
    kv8 = ctx_sum * 2 * Hkv * (D + 4) * L    # codes and one f32 scale per row
    bytes8 = sb["layers"] + sb["lm_head"] + kv8
    bytes16 = sb["total"]
    peaks = measured_peaks()
    line = {"metric": "A8W8 batched decode step over an INT8 KV cache (ms/step, 40 layers, bs=16, "
                      "fixed contexts 64..4096)",
            "value": ms[True], "unit": "ms/step", "n_gpus": 1, "steps": n, "warmup": args.warmup,
            "ms_per_step": ms[True], "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None,
            "dtype": "int8 x int8 -> int32, f32 dequant, int8 KV codes x f32 row scales",
            "data": "synthetic (seeded random-init weights; random KV codes and row scales)",
            "config": {"workload": "qwen3_14b_a8w8_batched_decode_b16_int8_kv", "batch": B,
                       "layers": L, "ctx_sum": ctx_sum, "page_size": page,
                       "l2": "inputs larger than L2 (13.2 GB of weights + KV per step)"},
            "tokens_per_s": job_rate(B, ms[True], 1),
            "step_bytes": bytes8, "step_hbm_gbs": bytes8 / (ms[True] * 1e-3) / 1e9,
            "step_frac_of_peak": bytes8 / (ms[True] * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "bf16_kv": {"ms_per_step": ms[False], "step_bytes": bytes16,
                        "step_hbm_gbs": bytes16 / (ms[False] * 1e-3) / 1e9},
            "kv_bytes": {"int8": kv8, "bf16": sb["kv"]},
            "e2e": None, "clocks": clock_runs, "device_errors": errs}
    print(json.dumps(line), flush=True)


PREFILL_SEQS, PREFILL_LEN = 4, 512
PREFILL_WORKLOAD = "qwen3_14b_a8w8_prefill_chunk_4x512"
PREFILL_METRIC = "A8W8 prefill chunk through one layer (ms, 4 x 512 tokens)"
# Dense FP16/BF16 tensor rate: the prefill projections multiply exact FP16
# images of the INT8 codes; MEASURED_PEAKS.json holds the bf16 figure (same
# nominal rate as fp16).
def tensor_peak() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"tflops": d["bf16_tflops"], "source": "measured (bf16 dense, MEASURED_PEAKS.json)"}
    return {"tflops": 1900.0, "source": "fallback (bf16 dense)"}


def run_prefill(args, cfg):
    """One layer over the pages' prefill chunk: 4 sequences x 512 tokens."""
    import torch
    import w8a8_quantized_decode_gb300 as a8w8

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    a8w8.build()
    cfg = dict(cfg, num_layers=1)
    page = cfg["page_size"]
    Hkv, D, H = cfg["num_kv_heads"], cfg["head_dim"], cfg["hidden"]
    M = PREFILL_SEQS * PREFILL_LEN
    bt_seq, nblk = synth.paged_layout(SEED + 31, [PREFILL_LEN] * PREFILL_SEQS, page,
                                      spare_blocks=1)
    rows = np.repeat(np.arange(PREFILL_SEQS), PREFILL_LEN)
    pos = np.tile(np.arange(PREFILL_LEN), PREFILL_SEQS)
    bt = bt_seq[rows].astype(np.int32)
    ctx = (pos + 1).astype(np.int32)
    slots = (bt_seq[rows, pos // page] * page + pos % page).astype(np.int32)
    w = synth.t_layer_weights(cfg, SEED, 0, device)
    gen = torch.Generator(device=device)
    gen.manual_seed(SEED + 32)
    hidden = torch.randn((M, H), generator=gen, device=device).to(torch.bfloat16)
    kc = torch.zeros((nblk * page, Hkv, D), dtype=torch.bfloat16, device=device)
    vc = torch.zeros_like(kc)
    rope = a8w8.a8w8_rope_table(bt.shape[1] * page, D, cfg["rope_theta"], device=device)
    ws = a8w8.alloc_workspace(cfg, M, bt.shape[1], device=device)
    d_bt, d_ctx, d_slot = (torch.from_numpy(x).to(device) for x in (bt, ctx, slots))
    h0 = hidden.clone()
    stream = torch.cuda.Stream(device)
    times = []
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            hidden.copy_(h0)
            a8w8.a8w8_prefill_layer(w, cfg, hidden, d_slot, d_bt, d_ctx, kc, vc, rope, ws,
                                    stream=stream)
        stream.synchronize()
        gpu_uuid = None
        try:
            gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            pass
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        with ClockSampler(gpu_uuid) as clocks:
            for _ in range(args.steps):
                hidden.copy_(h0)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                a8w8.a8w8_prefill_layer(w, cfg, hidden, d_slot, d_bt, d_ctx, kc, vc, rope, ws,
                                        stream=stream)
                e1.record(stream)
                e1.synchronize()
                times.append(e0.elapsed_time(e1))
        errs = a8w8.read_device_errors(stream)
        # the dominant contraction alone: the Gate/Up GEMM's exact INT32
        # product (tcgen05) on the chunk's quantised rows, CUDA events on
        # `stream` around `reps` back-to-back launches
        xq = torch.randint(-127, 128, (M, H), dtype=torch.int8, device=device)
        acc = torch.empty((M, 2 * cfg["intermediate"]), dtype=torch.int32, device=device)
        scratch = torch.empty((M * H,), dtype=torch.float16, device=device)
        for _ in range(2):
            a8w8.a8w8_matmul_i8(xq, w["w_gate_up"], out=acc, scratch=scratch, stream=stream)
        reps = 5
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        stream.synchronize()
        g0.record(stream)
        for _ in range(reps):
            a8w8.a8w8_matmul_i8(xq, w["w_gate_up"], out=acc, scratch=scratch, stream=stream)
        g1.record(stream)
        g1.synchronize()
        gu_ms = g0.elapsed_time(g1) / reps
        del acc, scratch
    ms = sum(times) / len(times)
    ms = max_over_ranks(ms, device)
    gu_flop = 2.0 * M * 2 * cfg["intermediate"] * H
    gu_tflops = gu_flop / (gu_ms * 1e-3) / 1e12
    ops = 2.0 * M * (cfg["hidden"] * ((cfg["num_q_heads"] + 2 * Hkv) * D) +
                      cfg["num_q_heads"] * D * cfg["hidden"] + 2 * cfg["intermediate"] * cfg["hidden"]
                      + cfg["intermediate"] * cfg["hidden"])
    attn_flops = 4.0 * PREFILL_SEQS * (PREFILL_LEN * (PREFILL_LEN + 1) / 2) * cfg["num_q_heads"] * D
    tops = ops / (ms * 1e-3) / 1e12
    tpk = tensor_peak()
    # per layer: 3 row quantisations (input norm, attention output, act; the
    # post-attention norm is the fourth), 4 GEMMs + 1 more for the down
    # projection's second K half, 4 epilogues, the KV pre-pass, attention
    n_launch = 4 + 5 + 4 + 1 + 1
    if rank == 0:
        line = {
            "metric": PREFILL_METRIC, "value": ms, "unit": "ms/chunk-layer", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8 x int8 -> int32, f32 dequant, bf16 activations",
            "data": "synthetic (seeded random-init weights and hidden states on the device)",
            "config": {"workload": PREFILL_WORKLOAD, "sequences": PREFILL_SEQS,
                       "tokens_per_sequence": PREFILL_LEN, "M": M, "layers": 1,
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "tokens_per_s": job_rate(M, ms, world),
            "int8_ops_per_s_e12": tops,
            "attention_flop": attn_flops,
            "layer_tflops": tops, "layer_frac_of_tensor_peak": tops / tpk["tflops"],
            "roofline": {"bound": "tensor",
                         "kernel": "Gate/Up GEMM, exact INT32 product of 2048 x 5120 by "
                                   "34816 x 5120 INT8 (gemm_tc_kernel: tcgen05.mma kind::f16 on "
                                   "exact FP16 images, TMA-fed, TMEM accumulators)",
                         "achieved": gu_tflops, "peak": tpk["tflops"], "unit": "TFLOP/s",
                         "frac": gu_tflops / tpk["tflops"], "traffic": None,
                         "flop_per_launch": gu_flop, "ms_per_launch": gu_ms,
                         "peak_source": tpk["source"]},
            "e2e": None,
            "gpu_launches": n_launch * args.steps,
            "clocks": clocks.summary(),
            "device_errors": errs,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


TTFT_LEN = 512
TTFT_WORKLOAD = "qwen3_14b_a8w8_ttft_prompt512"


def run_ttft(args, cfg):
    """Time to first token: one 512-token prompt through the 40 layers as one
    prefill chunk, then the final norm, LM head and argmax on its last row
    (a8w8_prefill_step); `e2e` adds the host->device copy of the prompt's
    inputs and the device->host read of the token (rank 0 only)."""
    import torch
    import w8a8_quantized_decode_gb300 as a8w8

    rank, world, local = dist_env()
    if rank != 0:
        return
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    a8w8.build()
    P, page = TTFT_LEN, cfg["page_size"]
    Hkv, D, L = cfg["num_kv_heads"], cfg["head_dim"], cfg["num_layers"]
    bt_seq, nblk = synth.paged_layout(SEED + 60, [P + 1], page, spare_blocks=1)
    pos = np.arange(P)
    bt = np.repeat(bt_seq, P, axis=0).astype(np.int32)
    ctx = (pos + 1).astype(np.int32)
    slots = (bt_seq[0, pos // page] * page + pos % page).astype(np.int32)
    tok = synth.prompt_ids(SEED + 61, P, cfg["vocab"])
    model = build_model(cfg, device)
    kc = [torch.zeros((nblk * page, Hkv, D), dtype=torch.bfloat16, device=device) for _ in range(L)]
    vc = [torch.zeros_like(k) for k in kc]
    rope = a8w8.a8w8_rope_table(bt.shape[1] * page, D, cfg["rope_theta"], device=device)
    ws = a8w8.alloc_workspace(cfg, P, bt.shape[1], device=device)
    host = {n: torch.from_numpy(x).pin_memory() for n, x in
            (("tok", tok), ("slot", slots), ("bt", bt), ("ctx", ctx))}
    dev = {n: t.to(device) for n, t in host.items()}
    last = torch.tensor([P - 1], dtype=torch.int32, device=device)
    nxt = torch.empty(1, dtype=torch.int32, device=device)
    nxt_host = torch.empty(1, dtype=torch.int32).pin_memory()
    stream = torch.cuda.Stream(device)

    def prefill():
        a8w8.a8w8_prefill_step(model, cfg, dev["tok"], dev["slot"], dev["bt"], dev["ctx"], kc, vc,
                               rope, ws, last, nxt, stream=stream)

    gpu_uuid = None
    try:
        gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass
    times, e2e_times = [], []
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            prefill()
        stream.synchronize()
        with ClockSampler(gpu_uuid) as clocks:
            for _ in range(args.steps):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                prefill()
                e1.record(stream)
                e1.synchronize()
                times.append(e0.elapsed_time(e1))
            for _ in range(args.steps):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for n in host:
                    dev[n].copy_(host[n], non_blocking=True)
                prefill()
                nxt_host.copy_(nxt, non_blocking=True)
                e1.record(stream)
                e1.synchronize()
                e2e_times.append(e0.elapsed_time(e1))
        errs = a8w8.read_device_errors(stream)
    ms = sum(times) / len(times)
    e2e_ms = sum(e2e_times) / len(e2e_times)
    H, I, Hq = cfg["hidden"], cfg["intermediate"], cfg["num_q_heads"]
    ops = 2.0 * P * L * (H * ((Hq + 2 * Hkv) * D) + Hq * D * H + 3 * I * H) + 2.0 * H * cfg["vocab"]
    tops = ops / (ms * 1e-3) / 1e12
    tpk = tensor_peak()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    # embed; per layer 15 (as the prefill layer); gather; LM head
    n_launch = 1 + 15 * L + 1 + 1
    line = {"metric": "A8W8 time to first token (ms, 512-token prompt, 40 layers, greedy)",
            "value": ms, "unit": "ms", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": False, "vs_baseline": None,
            "dtype": "int8 x int8 -> int32 (fp16 tensor-core images), f32 dequant, bf16 activations",
            "data": "synthetic (seeded random-init weights; empty KV history)",
            "config": {"workload": TTFT_WORKLOAD, "prompt_tokens": P, "layers": L,
                       "page_size": page, "l2": "inputs larger than L2 (14.8 GB of weights)"},
            "tokens_per_s": P / (ms * 1e-3),
            "roofline": {"bound": "tensor",
                         "kernel": "whole prefill (projections as tcgen05 GEMMs on exact "
                                   "images of the INT8 codes, epilogues, attention, LM head row)",
                         "achieved": tops, "peak": tpk["tflops"], "unit": "TFLOP/s",
                         "frac": tops / tpk["tflops"], "traffic": None, "peak_source": tpk["source"]},
            "e2e": {"value": e2e_ms, "unit": "ms", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4},
            "gpu_launches": n_launch * args.steps,
            "clocks": clocks.summary(), "device_errors": errs}
    print(json.dumps(line), flush=True)


LAYER_B1_VARIANTS = {
    "layer_b1": ("a8w8", "A8W8 decode layer, batch 1, context 256 (us per layer)",
                 "qwen3_14b_a8w8_layer_b1_ctx256",
                 "int8 x int8 -> int32, f32 dequant, bf16 activations"),
    "layer_b1_i8kv": ("i8kv", "A8W8 decode layer, INT8 KV cache, batch 1, context 256 (us per layer)",
                      "qwen3_14b_a8w8_i8kv_layer_b1_ctx256",
                      "int8 x int8 -> int32, f32 dequant, int8 KV codes x f32 row scales"),
    "layer_b1_bf16": ("bf16", "BF16 decode layer, batch 1, context 256 (us per layer)",
                      "qwen3_14b_bf16_layer_b1_ctx256",
                      "bf16 x bf16 products, f32 sums, bf16 activations"),
}


def run_layer_b1(args, cfg):
    """One decode layer, batch 1, 255 cached tokens + the decoded one (context
    256, pages of 128), the layer's weights rotated over 4 copies so that L2
    (129 MB) cannot serve a repeat (rank 0 only). Variants: the A8W8 layer
    (BF16 KV cache), the A8W8 layer over the INT8 KV cache, the BF16 layer."""
    import torch
    import w8a8_quantized_decode_gb300 as a8w8

    rank, world, local = dist_env()
    if rank != 0:
        return
    variant, metric, workload, dtype = LAYER_B1_VARIANTS[args.workload]
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    a8w8.build()
    cfg = dict(cfg, num_layers=1)
    page, ctx = cfg["page_size"], 256
    Hkv, D, H = cfg["num_kv_heads"], cfg["head_dim"], cfg["hidden"]
    if variant == "bf16":
        copies = [synth.t_bf16_layer_weights(cfg, SEED + 50 + c, 0, device) for c in range(4)]
        # every matrix and norm weight in BF16, no scales
        weight_bytes = sum(2 * int(np.prod(shape)) for kind, shape in synth.weight_shapes(cfg).values()
                           if kind != "f32")
    else:
        copies = [synth.t_layer_weights(cfg, SEED + 50 + c, 0, device) for c in range(4)]
        weight_bytes = synth.layer_weight_bytes(cfg)
    bt_np, nblk = synth.paged_layout(SEED + 51, [ctx], page, spare_blocks=1)
    gen = torch.Generator(device=device)
    gen.manual_seed(SEED + 52)
    if variant == "i8kv":
        kc, ks = synth.t_i8_kv_history(SEED + 53, nblk * page, Hkv, D, device)
        vc, vs = synth.t_i8_kv_history(SEED + 55, nblk * page, Hkv, D, device)
        kv_bytes = ctx * 2 * Hkv * (D + 4)
    else:
        kc = torch.randn((nblk * page, Hkv, D), generator=gen, device=device).to(torch.bfloat16)
        vc = torch.randn((nblk * page, Hkv, D), generator=gen, device=device).to(torch.bfloat16)
        kv_bytes = ctx * 2 * Hkv * D * 2
    hidden = torch.randn((1, H), generator=gen, device=device).to(torch.bfloat16)
    h0 = hidden.clone()
    bt = torch.from_numpy(bt_np).to(device)
    cl = torch.tensor([ctx], dtype=torch.int32, device=device)
    sl = torch.from_numpy(synth.slots_for(bt_np, [ctx - 1], page)).to(device)
    rope = a8w8.a8w8_rope_table(bt_np.shape[1] * page, D, cfg["rope_theta"], device=device)
    ws = a8w8.alloc_workspace(cfg, 1, bt_np.shape[1], device=device)
    stream = torch.cuda.Stream(device)

    def layer(w):
        if variant == "i8kv":
            a8w8.a8w8_decode_layer_i8kv(w, cfg, hidden, sl, bt, cl, kc, vc, ks, vs, rope, ws,
                                        stream=stream)
        elif variant == "bf16":
            a8w8.bf16_decode_layer(w, cfg, hidden, sl, bt, cl, kc, vc, rope, ws, stream=stream)
        else:
            a8w8.a8w8_decode_layer(w, cfg, hidden, sl, bt, cl, kc, vc, rope, ws, stream=stream)

    n = max(args.steps, 8)
    with torch.cuda.stream(stream):
        g = torch.cuda.CUDAGraph()
        # one graph replay = n layer calls over the 4 rotating copies
        for _ in range(2):
            for i in range(4):
                layer(copies[i])
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                layer(copies[i % 4])
        for _ in range(args.warmup):
            hidden.copy_(h0)
            g.replay()
        stream.synchronize()
        gpu_uuid = None
        try:
            gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            pass
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        reps = 10    # ~35 ms timed, so that the clock sampler sees the run
        with ClockSampler(gpu_uuid) as clocks:
            hidden.copy_(h0)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
            e1.synchronize()
        errs = a8w8.read_device_errors(stream)
    us = e0.elapsed_time(e1) * 1000.0 / (n * reps)
    layer_bytes = weight_bytes + kv_bytes
    peaks = measured_peaks()
    line = {"metric": metric, "value": us,
            "unit": "us/layer", "n_gpus": 1, "steps": n * reps, "warmup": args.warmup,
            "higher_is_better": False, "vs_baseline": None, "dtype": dtype,
            "data": "synthetic (seeded random-init weights, 4 rotating copies; random context K/V)",
            "config": {"workload": workload, "batch": 1, "context": ctx, "weight_copies": 4,
                       "l2": "weights rotated over 4 copies, larger than L2"},
            "layer_bytes": layer_bytes, "hbm_gbs": layer_bytes / (us * 1e-6) / 1e9,
            "frac_of_peak": layer_bytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"],
            "clocks": clocks.summary(), "device_errors": errs}
    print(json.dumps(line), flush=True)


def run_sample(args, cfg):
    """Device-side sampling over the 151936-token vocabulary (rank 0 only):
    microseconds per call at batch 1 and 16, greedy, temperature and top-p."""
    import torch
    import w8a8_quantized_decode_gb300 as a8w8

    rank, world, local = dist_env()
    if rank != 0:
        return
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    a8w8.build()
    V = cfg["vocab"]
    gen = torch.Generator(device=device)
    gen.manual_seed(SEED + 41)
    res = {}
    for B in (1, 16):
        logits = torch.randn((B, V), generator=gen, device=device) * 2.0
        out = torch.empty(B, dtype=torch.int32, device=device)
        ws = torch.empty(a8w8.lib().a8w8_sample_workspace_bytes(B, V), dtype=torch.uint8,
                         device=device)
        for name, T, p in (("greedy", 0.0, 1.0), ("temperature", 0.7, 1.0), ("top_p", 0.7, 0.9)):
            for s in range(args.warmup):
                a8w8.a8w8_sample(logits, T, p, 1, s, out=out, ws=ws)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for s in range(args.steps):
                a8w8.a8w8_sample(logits, T, p, 1, s, out=out, ws=ws)
            e1.record()
            e1.synchronize()
            res[f"b{B}_{name}_us"] = e0.elapsed_time(e1) * 1000.0 / args.steps
    line = {"metric": "device sampling over 151936 logits (us per call)",
            "value": res["b1_top_p_us"], "unit": "us/call", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": False, "vs_baseline": None,
            "dtype": "f32 logits, two-float softmax masses, f32 Gumbel keys",
            "data": "synthetic N(0, 2^2) logits", "config": {"workload": "sample", "vocab": V},
            "detail": res}
    print(json.dumps(line), flush=True)


def cpu_baseline(model, cfg):
    """The oracle on a bounded sample: decode steps until about 20 s of CPU time."""
    import torch
    hm = host_model(model)
    import oracle
    oracle.build()
    times, threads = time_oracle_steps(hm, cfg, n_steps=8, budget_s=20.0)
    del hm
    return {"value": 1000.0 * sum(times) / len(times), "unit": "ms/token", "cores": threads,
            "kind": "oracle", "host": host_cpu(),
            "sample": f"{len(times)} oracle decode steps of the same workload (40 layers + LM "
                      f"head, batch 1, contexts {PROMPT_LEN + 1}..{PROMPT_LEN + len(times)})"}


def build_parser() -> argparse.ArgumentParser:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["decode_b1", "decode_b1_sampled", "batched16",
                                           "batched16_i8kv", "prefill", "ttft", "sample",
                                           *LAYER_B1_VARIANTS],
                    default="decode_b1")
    ap.add_argument("--layers", type=int, default=40,
                    help="layers of the model (fewer only for profiling captures)")
    return ap


def main():
    args = build_parser().parse_args()
    if args.steps is None:
        args.steps = {"batched16": 32, "batched16_i8kv": 16, "prefill": 5, "ttft": 5, "sample": 20,
                      **{w: 40 for w in LAYER_B1_VARIANTS}}.get(args.workload, 48)
    if args.warmup < 3:
        raise SystemExit("warmup must be >= 3")
    cfg = dict(synth.QWEN3_14B, num_layers=args.layers)
    if args.impl == "reference":
        run_reference(args, cfg)
    elif args.workload == "batched16":
        run_batched(args, cfg)
    elif args.workload == "batched16_i8kv":
        run_batched_i8kv(args, cfg)
    elif args.workload == "ttft":
        run_ttft(args, cfg)
    elif args.workload == "prefill":
        run_prefill(args, cfg)
    elif args.workload == "sample":
        run_sample(args, cfg)
    elif args.workload == "decode_b1_sampled":
        run_sampled(args, cfg)
    elif args.workload in LAYER_B1_VARIANTS:
        run_layer_b1(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
