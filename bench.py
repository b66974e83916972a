"""Benchmark of the stage forward on GB300.

Default workload: the dense 8B-shape decoder (32 blocks, hidden 4096, 32 q / 8 kv heads x
128, SwiGLU 14336, vocab 32000, int8 block-32 weights) as 2 stages split 16/16 on one GPU,
batch-1 greedy decode at context 2048.  A step = one token through both stages, the
final norm, the readout and the greedy argmax (every row of the hot path).

value : decode tok/s, device-timed (CUDA events on the stages' stream) over K graph-replayed
        steps with everything resident in HBM; weights (7.5 GB) exceed L2, so every step
        streams them from HBM.
e2e   : the same through the C ABI with host buffers (stage_pipeline_step per token: host
        seq/pos/token arrays copied in, the greedy token read back each step).
roofline: bytes per token (weights once + KV at the context) / step time against the
        measured HBM peak; the dominant kernel is timed on its own in a second pass.
prefill: on the same dense stages, 4 prompts x 512 tokens as one step (every projection a
        tcgen05 GEMM with bf16 operands), prefill tok/s and the gate/up GEMM's TFLOP/s
        against the measured bf16 peak.
moe_decode, batched_70b_decode: the MoE 40-block decoder (2 stages 21/19, context 4096) and
        the 70B-shape batched decode (4 stages of 20 blocks, 64 ragged sequences), each as a
        record of the same line with its own roofline, e2e and clocks.
--impl reference: the CPU oracle on the host cores, on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

# workloads: the dense 8B-shape decoder (default) and the 40-block MoE decoder
WORKLOADS = {
    1: dict(context=2048, bounds=[0, 16, 32],
            name="dense 8B-shape decode, 32 blocks as 2 stages 16/16, batch 1, context 2048"),
    2: dict(context=4096, bounds=[0, 21, 40],
            name="MoE 40-block decode (128 experts top-8), 2 stages 21/19, batch 1, context 4096"),
    4: dict(context=None, bounds=[0, 20, 40, 60, 80], seqs=64,
            name="dense 70B-shape batched decode, 80 blocks as 4 stages 20/20/20/20, 64 sequences with KV "
                 "lengths uniform in 128-4096"),
}
CFG_ID = 1
CONTEXT = 2048
# the prefill workload: the dense 8B-shape stages, a batch of 4 seeded prompts of 512 tokens
PREFILL = dict(seqs=4, prompt=512, min_tokens=64,
               name="dense 8B-shape prefill, 2 stages 16/16, 4 prompts x 512 tokens in one step, "
                    "bf16 tcgen05 GEMMs with int8 block-32 weights dequantised in shared memory")
# DRAM bytes (read + write) per launch of the dominant kernel, the persistent stage decode:
# an ncu capture of one block in the same launch configuration (the bytes of a block do not
# depend on its index), scaled by the 16 blocks of a launch of the dense workload.  The MoE
# kernel has changed since its capture: its traffic is reported as unknown.
TRAFFIC = {1: 3_907_534_848}


def dist_env():
    """(rank, world size, local rank) from the launcher's environment (1 process by default)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(world, backend):
    """The process group of a multi-replica run (None for one process)."""
    if world <= 1:
        return None
    import torch.distributed as dist
    dist.init_process_group(backend)
    return dist


def max_over_ranks(x, dist, device=None):
    """The maximum of x over all ranks: a replica run is as slow as its slowest replica."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank, seconds, world):
    """Whole-job throughput: every rank processed units_per_rank in at most `seconds`."""
    return units_per_rank * world / seconds


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return {}


def bytes_per_token(model, context):
    """Algorithmic bytes of one decode token: every weight byte the token needs once (1 B
    int8 + 2 B per 32-weight scale = 1.0625 B/param; for MoE only the router and the top-k
    experts) plus the fp16 K and V rows of every position attended."""
    H, D = model.hidden, model.head_dim
    per_layer = (model.q_dim + 2 * model.kv_dim) * H + H * model.q_dim
    if model.is_moe:
        per_layer += model.n_experts * H + model.top_k * 3 * model.expert_ffn * H
    else:
        per_layer += 3 * model.ffn * H
    params = per_layer * model.n_layers + model.vocab * H  # readout; the embedding reads one row
    w = params * 1.0625 + H * 1.0625
    kv = model.n_layers * 2 * model.n_kv_heads * context * D * 2
    return w, kv


class ClockSampler:
    def __init__(self, period_s=0.2):
        self.samples, self.period, self._stop = [], period_s, threading.Event()
        self._t = None

    def start(self):
        def run():
            q = ("--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap")
            while not self._stop.is_set():
                try:
                    out = subprocess.run(["nvidia-smi", q, "--format=csv,noheader,nounits", "-i", "0"],
                                         capture_output=True, text=True, timeout=5).stdout.strip()
                    if out:
                        self.samples.append([x.strip() for x in out.split(",")])
                except Exception:
                    pass
                self._stop.wait(self.period)
        self._t = threading.Thread(target=run, daemon=True)
        self._t.start()

    def stop(self):
        self._stop.set()
        if self._t:
            self._t.join(timeout=10)
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if len(s) > 2 + i and "Active" in s[2 + i]
                          and "Not" not in s[2 + i]})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


def build_gpu_pipeline(model, bounds, max_seq_len, max_tokens, max_seqs=1, gemm_bf16_min_tokens=0):
    from layer_range_stage_gb300.pipeline import StagePipeline
    return StagePipeline(model, bounds, lambda l: synth.layer_weights(model, l),
                         lambda a, b: synth.stage_weights(model, a, b, with_layers=False),
                         max_seqs=max_seqs, max_seq_len=max_seq_len, max_tokens=max_tokens,
                         gemm_bf16_min_tokens=gemm_bf16_min_tokens)


def gemm_flops_per_token(model):
    """2 x the projection weights one token multiplies (readout excluded)."""
    H = model.hidden
    per_layer = (model.q_dim + 2 * model.kv_dim) * H + H * model.q_dim + 3 * model.ffn * H
    return 2.0 * per_layer * model.n_layers


def run_prefill(gp, model, warm=2, reps=3):
    """Prefill steps of PREFILL's batch, each from empty caches; returns the prefill fields."""
    import torch
    import layer_range_stage_gb300 as L
    ns, plen = PREFILL["seqs"], PREFILL["prompt"]
    T = ns * plen
    toks = np.concatenate([synth.prompt_tokens(model, 100 + s, plen) for s in range(ns)])
    seq, pos = np.repeat(np.arange(ns), plen), np.tile(np.arange(plen), ns)
    rows = np.arange(1, ns + 1) * plen - 1
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for i in range(warm + reps + 1):
        for st in gp.stages:
            L.stage_reset(st)
        timed_kernel = i == warm + reps
        if timed_kernel:  # one more step with events around every gate/up GEMM
            gp.kernel_timing(True)
        torch.cuda.synchronize()
        e0.record(stream)
        gp.step(True, seq, pos, toks, rows=rows)
        e1.record(stream)
        torch.cuda.synchronize()
        if warm <= i < warm + reps:
            times.append(e0.elapsed_time(e1))
    k_us, k_n = gp.kernel_time()
    gp.kernel_timing(False)
    for st in gp.stages:
        L.stage_reset(st)
    ms = float(np.mean(times))
    peak = measured_peaks().get("bf16_tflops")
    k_flops = 2.0 * T * 2 * model.ffn * model.hidden
    k_tf = k_flops / (k_us * 1e-6) / 1e12 if k_us else None
    step_tf = gemm_flops_per_token(model) * T / (ms * 1e-3) / 1e12
    return {"value": round(T * 1000.0 / ms, 1), "unit": "tok/s", "ms_per_step": round(ms, 3), "steps": reps,
            "warmup": warm, "tokens_per_step": T, "workload": PREFILL["name"],
            "dtype": "bf16 operands, f32 accumulation",
            "roofline": {"bound": "tensor", "achieved": round(k_tf, 1) if k_tf else None, "peak": peak,
                         "unit": "TFLOP/s", "frac": round(k_tf / peak, 4) if (k_tf and peak) else None,
                         "traffic": None, "kernel": "FFN gate/up tcgen05 GEMM (SwiGLU epilogue)",
                         "flops_per_launch": k_flops, "mean_launch_us": round(k_us, 2), "launches_timed": k_n,
                         "peak_source": "measured burst (MEASURED_PEAKS.json bf16_tflops)" if peak else "fallback"},
            "step_roofline": {"bound": "tensor", "achieved": round(step_tf, 1), "peak": peak, "unit": "TFLOP/s",
                              "frac": round(step_tf / peak, 4) if peak else None,
                              "flops_per_step": gemm_flops_per_token(model) * T}}


def run_gpu(args, config=None, dist=None):
    """One decode workload (cfg1 dense, cfg2 MoE): the bench line's fields, as a dict."""
    import torch
    import layer_range_stage_gb300 as L  # noqa: F401

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    config = config or args.config
    wl = WORKLOADS[config]
    model = synth.CONFIGS[config]
    bounds = wl["bounds"]
    context = args.context or wl["context"]
    if args.layers:  # reduced depth: profiling of a small case only, never a bench line
        model = synth.reduced(model, args.layers)
        bounds = [0, args.layers // 2, args.layers] if args.layers > 1 else [0, 1]
    steps, warmup = args.steps, args.warmup
    max_len = context + warmup + 2 * steps + 16
    t_build = time.time()
    dense = not model.is_moe
    if dense:  # room for the prefill batch; calls of >= 64 tokens run on the tensor cores
        gp = build_gpu_pipeline(model, bounds, max(max_len, PREFILL["prompt"]), max_tokens=PREFILL["seqs"] * PREFILL["prompt"],
                                max_seqs=PREFILL["seqs"], gemm_bf16_min_tokens=PREFILL["min_tokens"])
    else:
        gp = build_gpu_pipeline(model, bounds, max_len, max_tokens=512)
    build_s = time.time() - t_build
    prefill = run_prefill(gp, model) if (dense and not getattr(args, "no_prefill", False)) else None
    # prefill the seeded context in chunks of 512 tokens through the stages
    prompt = synth.prompt_tokens(model, rank, context)
    tok = None
    for c0 in range(0, context, 512):
        c1 = min(context, c0 + 512)
        tok = gp.step(True, np.zeros(c1 - c0), np.arange(c0, c1), prompt[c0:c1], rows=[c1 - c0 - 1])
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    # warm-up (captures the step graph), then K timed graph replays
    first = gp.generate([0], tok, warmup, use_graph=True)[-1]
    if dist:
        dist.barrier()
    clocks = ClockSampler()
    clocks.start()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    last = gp.generate([0], first, steps, use_graph=True)[-1]
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, "cuda")
    if dist:
        dist.barrier()
    ctx_mid = context + warmup + steps / 2
    w_bytes, kv_bytes = bytes_per_token(model, ctx_mid)
    ms_step = ms / steps
    tok_s = aggregate_rate(steps, ms * 1e-3, world)
    gbs = (w_bytes + kv_bytes) / (ms_step * 1e-3) / 1e9

    # the dominant kernel timed with CUDA events recorded around each of its launches inside
    # a second run of the same graph-replayed steps (events between kernels cost overlap, so
    # the headline number above comes from the run without them): on dense stages the
    # persistent decode kernel (one launch per stage per token; the mean over the stages'
    # launches)
    gp.kernel_timing(True)
    nxt = gp.generate([0], last, 4, use_graph=True)[-1]
    torch.cuda.synchronize()
    k_us, k_n = gp.kernel_time()
    gp.kernel_timing(False)
    last = nxt
    steps_extra = 4
    # e2e: stage_pipeline_step per token with host buffers (token read back every step)
    cur = context + warmup + steps + steps_extra
    tk = int(last[0])
    for _ in range(2):
        tk = int(gp.step(False, [0], [cur], [tk], rows=[0])[0])
        cur += 1
    torch.cuda.synchronize()
    n_e2e = max(4, steps // 2)
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        tk = int(gp.step(False, [0], [cur], [tk], rows=[0])[0])
        cur += 1
    e2e_s = time.perf_counter() - t0
    e2e = {"value": n_e2e * world / e2e_s, "unit": "tok/s", "h2d_bytes_per_step": 4 * (3 + 2 + 1),
           "d2h_bytes_per_step": 4, "steps": n_e2e}
    gp.close()

    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    H = model.hidden
    blocks = model.n_layers / (len(bounds) - 1)  # mean blocks per launch
    per_block = (model.q_dim + 2 * model.kv_dim) * H + H * model.q_dim
    if model.is_moe:  # the router once, the selected experts' gate/up and down rows
        kernel = (f"persistent decode of one stage (blocks {'/'.join(str(b - a) for a, b in zip(bounds, bounds[1:]))}: "
                  "QKV, attention, O, router + top-k, gathered expert gate/up, gathered expert down)")
        per_block += model.n_experts * H + model.top_k * 3 * model.expert_ffn * H
    else:
        kernel = "persistent decode of one stage (16 blocks: QKV, attention, O, gate/up, down)"
        per_block += 3 * model.ffn * H
    kv_block = 2 * model.n_kv_heads * (context + warmup + steps + 2) * model.head_dim * 2
    k_bytes = blocks * (per_block * 1.0625 + kv_block)
    k_gbs = k_bytes / (k_us * 1e-6) / 1e9 if k_us else None
    line = {
        "metric": "decode tok/s",
        "value": round(tok_s, 2), "unit": "tok/s", "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 (int8 block-32 weights, fp16 KV)", "data": "synthetic (seeded N(0,0.02) weights, seeded prompt)",
        "config": {"workload": wl["name"],
                   "parallelism": "replicas only" if world > 1 else "single GPU, 2 chained stages",
                   "l2": f"inputs larger than L2: {w_bytes / 1e9:.2f} GB of weights streamed per step"},
        "hbm_gbs_achieved": round(gbs, 1),
        "roofline": {"bound": "hbm", "achieved": round(k_gbs, 1) if k_gbs else None, "peak": peak, "unit": "GB/s",
                     "frac": round(k_gbs / peak, 4) if (peak and k_gbs) else None,
                     "traffic": TRAFFIC.get(config) if not (args.layers or args.context) else None,
                     "kernel": kernel,
                     "bytes_per_launch": round(k_bytes), "mean_launch_us": round(k_us, 3), "launches_timed": k_n,
                     "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak else "fallback"},
        "step_roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                          "frac": round(gbs / peak, 4) if peak else None,
                          "bytes_per_step": round(w_bytes + kv_bytes)},
        "e2e": e2e,
        "prefill": prefill,
        "clocks": clk,
        "gpu_launches": steps * (1 + (len(bounds) - 1) + 4),
        "build_s": round(build_s, 1),
    }
    if args.layers or args.context:
        line["config"]["profiling_case"] = f"{model.n_layers} blocks, context {context}: not the benchmark workload"
    return line


def batched_lens(nseq):
    """Seeded KV lengths of the batched workload: uniform in [128, 4096]."""
    return np.random.default_rng(4401).integers(128, 4097, nseq)


def run_batched(args, dist=None):
    """The 70B-shape batched decode: 4 stages of 20 blocks, 64 sequences of ragged context,
    one token per sequence per step (all stages, the final norm, the readout of the 64 rows
    and their argmax), on the float32 GEMV path and on the tensor-core path (bf16 operands,
    f32 accumulation: the stage's GEMM threshold set to the batch).  One seeded block of
    weights is loaded into every block (each block has its own device copy, so the bytes a
    step moves are those of 80 distinct blocks); every sequence's cache holds seeded fp16
    N(0, 1) K and V rows up to its length."""
    import torch
    from layer_range_stage_gb300 import binding as B
    from layer_range_stage_gb300.pipeline import StagePipeline

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    wl = WORKLOADS[4]
    model, bounds = synth.CONFIGS[4], wl["bounds"]
    if args.layers:  # reduced depth: profiling of a small case only, never a bench line
        model = synth.reduced(model, args.layers)
        bounds = sorted(set(int(round(x)) for x in np.linspace(0, args.layers, min(4, args.layers) + 1)))
    nseq = wl["seqs"]
    lens = batched_lens(nseq)
    seqs = np.arange(nseq)
    steps, warmup, n_timing, n_e2e = getattr(args, "batched_steps", None) or args.steps, args.warmup, 2, 4
    max_len = int(lens.max()) + warmup + steps + n_timing + n_e2e + 8
    t_build = time.time()
    block = synth.layer_weights(model, 0)
    kmax = int(lens.max())
    shape = (model.n_kv_heads, kmax, model.head_dim)
    size = int(np.prod(shape))
    kall = synth.normal_f32(synth.key(4400, 0, 0), 0, size, 1.0).reshape(shape).astype(np.float16)
    vall = synth.normal_f32(synth.key(4400, 0, 1), 0, size, 1.0).reshape(shape).astype(np.float16)
    kv = [(np.ascontiguousarray(kall[:, :n]), np.ascontiguousarray(vall[:, :n])) for n in lens]
    first = np.random.default_rng(4402).integers(0, model.vocab, nseq)
    H, D, F = model.hidden, model.head_dim, model.ffn
    per_layer = (model.q_dim + 2 * model.kv_dim) * H + H * model.q_dim + 3 * F * H
    w_bytes = (per_layer * model.n_layers + model.vocab * H + nseq * H) * 1.0625
    ctx = lens + warmup + steps / 2.0  # positions attended, mean over the timed steps
    kv_bytes = model.n_layers * 2 * model.n_kv_heads * D * 2 * float(np.sum(ctx + 1))
    peak = measured_peaks().get("hbm_gbs")
    stream = torch.cuda.current_stream()
    paths = {}
    for path, min_tok in (("f32", 0), ("bf16", nseq)):
        gp = StagePipeline(model, bounds, lambda l: block, lambda a, b: synth.stage_weights(model, a, b, with_layers=False),
                           max_seqs=nseq, max_seq_len=max_len, max_tokens=nseq, gemm_bf16_min_tokens=min_tok)
        try:
            for st, a, b in zip(gp.stages, bounds, bounds[1:]):
                for l in range(a, b):
                    for sq in range(nseq):
                        B.stage_write_kv(st, l, sq, 0, kv[sq][0], kv[sq][1])
                B.stage_commit(st, seqs, lens)
            torch.cuda.synchronize()
            tok = gp.generate(seqs, first, warmup, use_graph=True)[-1]
            if dist:
                dist.barrier()
            clocks = ClockSampler()
            clocks.start()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            last = gp.generate(seqs, tok, steps, use_graph=True)[-1]
            e1.record(stream)
            torch.cuda.synchronize()
            clk = clocks.stop()
            ms = max_over_ranks(e0.elapsed_time(e1), dist, "cuda")
            # the dominant kernel, the FFN gate/up launch of every block, timed with events
            # around each launch in a separate run of the same steps
            gp.kernel_timing(True)
            last = gp.generate(seqs, last, n_timing, use_graph=True)[-1]
            torch.cuda.synchronize()
            k_us, k_n = gp.kernel_time()
            gp.kernel_timing(False)
            # e2e: stage_pipeline_step with host arrays (64 ids, positions, tokens in; 64 tokens out)
            pos = lens + warmup + steps + n_timing
            tk = last
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for i in range(n_e2e):
                tk = gp.step(False, seqs, pos + i, tk, rows=seqs)
            e2e_s = time.perf_counter() - t0
        finally:
            gp.close()
        ms_step = ms / steps
        act = 4 if path == "f32" else 2  # the gate/up input and SwiGLU output: f32 rows, or bf16
        k_bytes = 2 * F * H * 1.0625 + nseq * H * act + nseq * F * act
        k_gbs = k_bytes / (k_us * 1e-6) / 1e9 if k_us else None
        paths[path] = {
            "value": round(aggregate_rate(nseq * steps, ms * 1e-3, world), 1), "ms_per_step": round(ms_step, 3),
            "hbm_gbs_achieved": round((w_bytes + kv_bytes) / (ms_step * 1e-3) / 1e9, 1),
            "roofline": {"bound": "hbm", "achieved": round(k_gbs, 1) if k_gbs else None, "peak": peak, "unit": "GB/s",
                         "frac": round(k_gbs / peak, 4) if (peak and k_gbs) else None, "traffic": None,
                         "kernel": ("FFN gate/up GEMV, 4 tokens per pass over the weights (SwiGLU epilogue)"
                                    if path == "f32" else
                                    "FFN gate/up tcgen05 small-call GEMM: 128 weight rows x 64 tokens, bf16 operands "
                                    "(SwiGLU epilogue)"),
                         "bytes_per_launch": round(k_bytes), "mean_launch_us": round(k_us, 2), "launches_timed": k_n,
                         "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak else "fallback"},
            "e2e": {"value": round(n_e2e * nseq * world / e2e_s, 1), "unit": "tok/s",
                    "h2d_bytes_per_step": 4 * 3 * nseq + 4 * nseq, "d2h_bytes_per_step": 4 * nseq, "steps": n_e2e},
            "clocks": clk,
            # per step: the embedding, per block 5 launches (QKV, attention, O, gate/up, down; the
            # tensor-core path adds 3 bf16 operand conversions), final norm, readout, argmax, advance
            "gpu_launches": steps * (1 + model.n_layers * (5 if path == "f32" else 8) + 4),
        }
    best = max(paths, key=lambda k: paths[k]["value"])
    b = paths[best]
    line = {
        "metric": "decode tok/s", "value": b["value"], "unit": "tok/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": b["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32 (int8 block-32 weights, fp16 KV)" if best == "f32" else
                 "bf16 GEMM operands, f32 accumulation (int8 block-32 weights, fp16 KV)",
        "data": "synthetic (one seeded N(0,0.02) block loaded into all 80; seeded fp16 N(0,1) KV rows)",
        "config": {"workload": wl["name"], "path": best,
                   "parallelism": "replicas only" if world > 1 else f"single GPU, {len(bounds) - 1} chained stages",
                   "l2": f"inputs larger than L2: {w_bytes / 1e9:.1f} GB of weights and {kv_bytes / 1e9:.1f} GB of KV "
                         "per step"},
        "hbm_gbs_achieved": b["hbm_gbs_achieved"],
        "roofline": b["roofline"],
        "step_roofline": {"bound": "hbm", "achieved": b["hbm_gbs_achieved"], "peak": peak, "unit": "GB/s",
                          "frac": round(b["hbm_gbs_achieved"] / peak, 4) if peak else None,
                          "bytes_per_step": round(w_bytes + kv_bytes)},
        "e2e": b["e2e"], "clocks": b["clocks"], "gpu_launches": b["gpu_launches"],
        "paths": paths, "wall_s": round(time.time() - t_build, 1),
    }
    if args.layers:
        line["config"]["profiling_case"] = f"{model.n_layers} blocks: not the benchmark workload"
    return line


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "cpu model")):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def blas_threads():
    """Threads the oracle's BLAS runs on: the thread-count variables OpenBLAS/OpenMP read,
    else every core (their default)."""
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    return os.cpu_count()


def cpu_baseline_one_thread(budget_s):
    """The same sample on one thread: a child process with the BLAS limited to one thread
    (the limit takes effect only when the BLAS starts)."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench.cpu_baseline(None, %r, one_thread_child=True)))" % (ROOT, budget_s))
    try:
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=600)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal
        return {"error": str(e)[:200]}


def oracle_sample_stage(max_new):
    """The oracle over 2 of the 32 blocks of the dense 8B shape (the first two, so it embeds and
    reads out), its KV filled with seeded fp16 values up to the decode context (the oracle's
    time does not depend on their values), room for max_new more tokens."""
    import oracle
    model = synth.CONFIGS[CFG_ID]
    n_blk = 2
    sub = synth.reduced(model, n_blk)
    w = synth.stage_weights(sub, 0, n_blk)
    st = oracle.Stage(sub, 0, n_blk, w, max_len=CONTEXT + max_new)
    rng = np.random.default_rng(0)
    st.k_cache[:] = rng.standard_normal(st.k_cache.shape).astype(np.float16)
    st.v_cache[:] = rng.standard_normal(st.v_cache.shape).astype(np.float16)
    return model, n_blk, st


def cpu_baseline(args, budget_s=None, one_thread_child=False):
    """The oracle as it stands, on a bounded sample: decode tokens through 2 of the 32
    blocks at context 2048 (KV filled with seeded fp16 values; the oracle's time does not
    depend on their values), repeated at successive positions until about budget_s seconds
    have passed, plus one readout; the mean block time is scaled to the 32-block token.
    Reported with the core count, the CPU model, the BLAS thread count and (unless this is
    the one-thread child) the same sample on one thread."""
    if budget_s is None:
        budget_s = getattr(args, "cpu_budget", 12.0)
    model, n_blk, st = oracle_sample_stage(max_new=64)
    cores = os.cpu_count()
    t_blocks, n_tok = 0.0, 0
    while n_tok < 2 or (t_blocks < budget_s and n_tok < 60):
        t0 = time.perf_counter()
        st.forward([0], [CONTEXT + n_tok], tokens=[1 + n_tok], cache_dequant=False)
        t_blocks += time.perf_counter() - t0
        n_tok += 1
    t0 = time.perf_counter()
    st.logits()
    t_head = time.perf_counter() - t0
    per_token = t_blocks / n_tok * model.n_layers / n_blk + t_head
    res = {"value": round(1.0 / per_token, 5), "unit": "tok/s", "cores": cores, "kind": "oracle",
           "threads": 1 if one_thread_child else blas_threads(), "cpu_model": cpu_model(),
           "sample": f"{n_tok} decode tokens through {n_blk} of {model.n_layers} blocks at context {CONTEXT}.., "
                     f"+ one readout; block time scaled x{model.n_layers // n_blk}; "
                     f"measured {t_blocks + t_head:.1f} s"}
    if not one_thread_child:
        one = cpu_baseline_one_thread(budget_s)
        res["one_thread"] = {k: one.get(k) for k in ("value", "unit", "threads", "sample", "error") if k in one}
    return res


def run_reference(args):
    """The reference arm: the oracle as it stands on the host cores, in steps like the GPU arm's:
    W untimed decode tokens, then K timed ones.  A step is one decode token at context 2048 on
    a bounded sample of the workload -- 2 of the 32 blocks, their time scaled to 32 -- plus that
    token's readout.  Under a multi-process launch rank 0 alone runs it and prints; the other
    ranks leave without work."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    model, n_blk, st = oracle_sample_stage(max_new=args.warmup + args.steps)
    scale = model.n_layers // n_blk
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        st.forward([0], [CONTEXT + i], tokens=[1 + i], cache_dequant=False)
        t1 = time.perf_counter()
        st.logits()
        t2 = time.perf_counter()
        if i >= args.warmup:
            times.append((t1 - t0) * scale + (t2 - t1))
    per_step = sum(times) / len(times)
    value = round(1.0 / per_step, 5)
    cb = {"value": value, "unit": "tok/s", "cores": os.cpu_count(), "threads": blas_threads(),
          "cpu_model": cpu_model(), "kind": "oracle",
          "sample": f"{args.steps} timed decode tokens (after {args.warmup} untimed) at context {CONTEXT}.. through "
                    f"{n_blk} of {model.n_layers} blocks, block time scaled x{scale}, each with its readout"}
    line = {"impl": "reference", "metric": "decode tok/s",
            "value": value, "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 1),
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOADS[1]["name"]},
            "cpu_baseline": cb, "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="reduced depth, for profiling small cases only")
    ap.add_argument("--context", type=int, default=0, help="decode context (default: the workload's)")
    ap.add_argument("--config", type=int, default=1, choices=sorted(WORKLOADS),
                    help="1: dense 8B-shape, 2: MoE, 4: dense 70B-shape batched decode (64 sequences)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work in the CPU baseline")
    ap.add_argument("--no-subrecords", action="store_true",
                    help="the dense decode line only (without the MoE and 70B-shape batched records)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
        return
    rank, world, _ = dist_env()
    dist = init_dist(world, "nccl")  # replicas only: the process group carries timing, no data
    if args.config == 4:
        line = run_batched(args, dist)
    else:
        line = run_gpu(args, args.config, dist)
        if args.config == 1 and not (args.layers or args.context or args.no_subrecords):
            # the other decode workloads, each a record of its own in the same line
            moe = run_gpu(argparse.Namespace(**{**vars(args), "no_prefill": True}), 2, dist)
            line["moe_decode"] = {k: moe[k] for k in ("metric", "value", "unit", "ms_per_step", "steps", "warmup",
                                                      "dtype", "config", "hbm_gbs_achieved", "roofline",
                                                      "step_roofline", "e2e", "clocks", "gpu_launches")}
            b70 = run_batched(argparse.Namespace(**{**vars(args), "batched_steps": max(3, args.steps // 4)}), dist)
            line["batched_70b_decode"] = {k: b70[k] for k in ("metric", "value", "unit", "ms_per_step", "steps",
                                                              "warmup", "dtype", "config", "hbm_gbs_achieved",
                                                              "roofline", "step_roofline", "e2e", "clocks",
                                                              "gpu_launches", "paths")}
    if rank == 0 and not args.no_cpu_baseline and world == 1 and args.config == 1:
        line["cpu_baseline"] = cpu_baseline(args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
