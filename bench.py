#!/usr/bin/env python
"""Benchmark of the lookahead decoding step (la_step) on GB300.

Workload (default): LLaMA-2-7B-shaped decoder, bf16, random N(0, 0.02)
weights from seed 0, batch 1, 256-token uniform prompt, N=5 W=15 G=15
(M = 121 step rows), greedy, 256 new tokens.

One timed "step" is one la_step call: candidate lookup, the forward pass over
the M rows, lm_head + argmax, verification, pool update, window slide and KV
commit, with the accepted tokens copied back to the host.  Each step is
bracketed by CUDA events on the handle's stream; W warm-up steps are not
timed.  The weights (13.2 GB) are far larger than L2, so no flush is needed.

JSON line (rank 0):
  value        committed tokens/s = accepted tokens / summed la_step time
  ms_per_step  mean la_step latency
  e2e          la_generate from a host prompt to host tokens (prefill included)
  roofline     dominant kernel (the tcgen05 projection GEMM): algorithmic
               bytes / event-timed launch time vs the measured HBM copy peak
  step_roofline (weight + KV bytes read per step) / la_step time vs the peak
  cpu_baseline the CPU oracle on the host cores, on a bounded sample
--impl reference: the CPU oracle alone, same metric, on bounded samples.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "la_step latency (ms) & committed tokens/s at 7B shape; % of HBM roofline per step"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=240)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama7b-bf16-greedy")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ncu", action="store_true",
                    help="profiling run: prefill + warm-up + timed steps only (no e2e, profiled pass or CPU baseline)")
    return ap.parse_args()


# ---------------------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            for k in ("hbm_gbs", "hbm_GBs", "hbm"):
                if k in d:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
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

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gemm_source_fp(read=None) -> str:
    """Fingerprint of the GEMM kernel sources with comments and blank lines
    removed, so that only a code change voids a traffic record."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "exact_decoding_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("gemm.cu", "la_common.cuh", "la_kernels.h"):
        text = read(f) if read else open(os.path.join(csrc, f)).read()
        if f == "la_kernels.h":
            # the shared header's GEMM section only (the rest declares other kernels)
            text = text[text.index("// " + "-" * 66 + " GEMMs"):text.index("// " + "-" * 66 + " elementwise")]
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(text.encode())
    return h.hexdigest()[:16]


def gemm_traffic():
    """DRAM bytes per k_gemm_tc2 launch from the committed ncu summary, or None
    when the kernel code changed since those counters were taken."""
    path = os.path.join(ROOT, "profiles", "k_gemm_tc2_traffic.txt")
    if not os.path.exists(path):
        return None
    rec = dict(line.split() for line in open(path) if line.strip())
    if gemm_source_fp() != rec.get("gemm_source_fp"):
        return None
    return float(rec["traffic_bytes_per_launch"])


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count()


def oracle_step_sample(weights, wl, prompt, layer: int):
    """Time the CPU oracle's forward for one lookahead step's M rows on a
    one-layer slice (layer `layer`, prefix = the prompt) and on a zero-layer
    slice (embedding + final norm + lm_head).  Returns (t_one_layer, t_head)."""
    import numpy as np
    from oracle import decoder, lookahead as la
    dims = weights["dims"]

    def sliced(layers):
        return {"dims": dataclasses.replace(dims, n_layers=len(layers)), "embed": weights["embed"],
                "layers": layers, "final_norm": weights["final_norm"], "lm_head": weights["lm_head"]}

    w1 = sliced([weights["layers"][layer]])
    w0 = sliced([])
    p = [int(t) for t in prompt]
    s = len(p)
    _, cache = decoder.forward(w1, p, np.arange(s), decoder.causal_mask(0, s), logit_rows=[s - 1])
    orc = la.Lookahead(w1, wl.N, wl.W, wl.G)
    orc.tokens = p + [p[-1]]
    orc.cache = cache
    orc.window = la.init_window(p, wl.N, wl.W, wl.seed)
    _, toks, pos, vis = orc.step_inputs()
    t0 = time.perf_counter()
    decoder.forward(w1, toks, pos, vis, cache=cache, logit_rows=orc.used)
    t1 = time.perf_counter()
    decoder.forward(w0, toks, pos, vis, cache=None, logit_rows=orc.used)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def extrapolated_step_seconds(t_layer_plus_head, t_head, n_layers):
    return n_layers * max(t_layer_plus_head - t_head, 0.0) + t_head


# ---------------------------------------------------------------------------- arms
def run_reference(args, wl):
    """CPU oracle arm: each step is a bounded sample (one decoder layer of the
    lookahead step plus the lm_head, extrapolated to all layers)."""
    import numpy as np
    import synth
    weights = synth.model_weights(wl.dims, wl.seed, layers=list(range(min(wl.dims.n_layers, args.steps + args.warmup))))
    prompt = synth.prompt(wl)
    times, walls = [], []
    for i in range(args.warmup + args.steps):
        layer = i % wl.dims.n_layers
        if weights["layers"][layer] is None:
            weights["layers"][layer] = synth.layer_weights(wl.dims, layer, wl.seed)
        tw = time.perf_counter()
        t1, t0 = oracle_step_sample(weights, wl, prompt, layer)
        tw = time.perf_counter() - tw
        if i >= args.warmup:
            times.append(extrapolated_step_seconds(t1, t0, wl.dims.n_layers))
            walls.append(tw)
    step_s = statistics.mean(times)
    # Tokens per step: a sampled step does not verify, so count the floor the
    # method guarantees (A = 1 committed token per step).  ms_per_step is the
    # wall time a sampled step really took here; the value scales the sample
    # to a whole step (all layers), reported as extrapolated_ms_per_step.
    value = 1.0 / step_s
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "committed tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.mean(walls) * 1e3, "extrapolated_ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, "prompt_len": wl.prompt_len, "N": wl.N, "W": wl.W,
                                        "G": wl.G, "rows_per_step": wl.M},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": "per step: oracle forward of the step's M rows through one decoder layer "
                                   "(256-token prefix) and through embedding+lm_head only; step time = "
                                   "n_layers x layer time + head time; 1 committed token per step (the floor)"},
        "e2e": {"value": value, "unit": "committed tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return line


def combine_ranks(accepted: float, total_ms: float, world: int, device: str = "cpu"):
    """Whole-job figures for N independent replicas (one per rank): committed
    tokens summed over ranks, timed region = the slowest rank's."""
    if world <= 1:
        return float(accepted), float(total_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(accepted)], dtype=torch.float64, device=device)
    m = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    dist.all_reduce(m, op=dist.ReduceOp.MAX)
    return float(t[0]), float(m[0])


def log(*a):
    print("[bench]", *a, file=sys.stderr, flush=True)


def run_ours(args, wl, rank, world, local_rank):
    import numpy as np
    import torch
    import synth
    import exact_decoding_gb300 as e

    torch.cuda.set_device(local_rank)
    t = time.perf_counter()
    weights = synth.lazy_model_weights(wl.dims, wl.seed)   # layers generated while they are uploaded
    prompt = synth.prompt(wl)
    dw = e.DeviceWeights(weights)
    log(f"weights generated and uploaded in {time.perf_counter() - t:.1f} s ({dw.nbytes() / 1e9:.1f} GB)")
    stream = torch.cuda.Stream()
    max_seq = wl.prompt_len + wl.new_tokens + wl.M + 8 * wl.N + 64
    kw = dict(temperature=wl.temperature, seed=wl.seed, prompt_as_reference=wl.prompt_as_reference)
    dec = e.Decoder(dw, wl.N, wl.W, wl.G, max_seq, stream=stream, **kw)

    def fresh():
        dec.prefill(prompt)

    def sync():
        stream.synchronize()
        torch.cuda.synchronize()

    # ---- end to end: la_generate, host prompt -> host tokens (one warm call first)
    toks, gen_steps, e2e_s, e2e_tps = [], 0, 0.0, None
    if not args.ncu:
        dec.generate(prompt, min(wl.new_tokens, 16))
        sync()
        t0 = time.perf_counter()
        toks, gen_steps = dec.generate(prompt, wl.new_tokens)
        sync()
        e2e_s = time.perf_counter() - t0
        e2e_tps = len(toks) / e2e_s
        gst = dec.stats()          # bytes the library copied in and out during that generation
    log(f"e2e: {len(toks)} tokens in {gen_steps} steps, {e2e_s:.3f} s")

    # ---- device-timed steps
    fresh()
    for _ in range(args.warmup):
        dec.step()
        if dec.stats()["generated"] + wl.N > wl.new_tokens:
            fresh()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    accepted, prefixes = 0, []
    launches0, launches = dec.stats()["kernel_launches"], 0
    if world > 1:
        torch.distributed.barrier()
    sync()
    with ClockSampler(local_rank) as clk:
        for i in range(args.steps):
            if dec.stats()["generated"] + wl.N > wl.new_tokens:
                launches += dec.stats()["kernel_launches"] - launches0
                fresh()        # untimed: a new generation of the same workload
                launches0 = 0
            prefixes.append(dec.stats()["prefix_len"])
            ev[i][0].record(stream)
            acc = dec.step()
            ev[i][1].record(stream)
            accepted += len(acc)
        sync()
    if world > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = sum(step_ms)
    log(f"timed: {args.steps} steps, {total_ms / args.steps:.3f} ms/step, {accepted} tokens")
    launches += dec.stats()["kernel_launches"] - launches0

    # ---- autoregressive baseline on this GPU: la_ar_step, same model and prompt
    ar_ms = None
    if not args.ncu:
        fresh()
        for _ in range(3):
            dec.ar_step()
        n_ar = 64
        ev_ar = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_ar)]
        sync()
        for i in range(n_ar):
            ev_ar[i][0].record(stream)
            dec.ar_step()
            ev_ar[i][1].record(stream)
        sync()
        ar_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_ar)
        log(f"autoregressive baseline: {ar_ms:.3f} ms/token")

    # ---- prefill, reported on its own: la_prefill of the host prompt (prompt
    # copy in, KV of every prompt token in 256-row passes, first token back)
    prefill_ms = None
    if not args.ncu:
        fresh()
        n_pf = 3
        ev_pf = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_pf)]
        sync()
        for i in range(n_pf):
            ev_pf[i][0].record(stream)
            fresh()
            ev_pf[i][1].record(stream)
        sync()
        prefill_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_pf)
        log(f"prefill: {len(prompt)} tokens in {prefill_ms:.3f} ms")

    # ---- profiled pass (events around every GEMM / attention launch)
    pdec = e.Decoder(dw, wl.N, wl.W, wl.G, max_seq, stream=stream, profile=True, **kw)
    if not args.ncu:
        pdec.prefill(prompt)
        for _ in range(min(args.steps, 16)):
            if pdec.stats()["generated"] + wl.N > wl.new_tokens:
                break
            pdec.step()
    pst = pdec.stats()
    pdec.close()
    log(f"profile: gemm {pst['gemm_ms']:.2f} ms / {pst['gemm_launches']} launches, "
        f"attn {pst['attn_ms']:.2f} ms / {pst['attn_launches']}, row-wise {pst['elem_ms']:.2f} ms, "
        f"speculation {pst['spec_ms']:.2f} ms, steps {pst['steps']}")

    accepted_all, max_ms = combine_ranks(accepted, total_ms, world, device="cuda")
    if rank != 0:
        dec.close()
        return None

    d = wl.dims
    act = 2 if d.dtype == "bf16" else 4
    weight_bytes = sum(t.numel() * t.element_size() for t in dw._keep if hasattr(t, "numel")) - d.vocab * d.d_model * act
    # Algorithmic K/V bytes per token: K and V of every layer at the weights'
    # element size (the cache's extra precision planes are not counted).
    kv_per_tok = 2 * d.n_layers * d.n_kv_heads * d.head_dim * act
    mean_P = statistics.mean(prefixes)
    step_bytes = weight_bytes + mean_P * kv_per_tok + wl.M * d.d_model * act + wl.N * kv_per_tok
    peak, peak_kind = peaks()
    ms_per_step = total_ms / args.steps
    step_gbs = step_bytes / (ms_per_step * 1e-3) / 1e9
    gemm_gbs = pst["gemm_bytes"] / (pst["gemm_ms"] * 1e-3) / 1e9 if pst["gemm_ms"] > 0 else None
    attn_gbs = pst["attn_bytes"] / (pst["attn_ms"] * 1e-3) / 1e9 if pst["attn_ms"] > 0 else None
    line = {
        "metric": METRIC, "value": accepted_all / (max_ms * 1e-3), "unit": "committed tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if d.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": wl.name, "prompt_len": wl.prompt_len, "N": wl.N, "W": wl.W, "G": wl.G,
                   "rows_per_step": wl.M, "new_tokens": wl.new_tokens, "temperature": wl.temperature,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2 ({weight_bytes / 1e9:.1f} GB of weights streamed per step)"},
        "step_stats": {"accepted_per_step": accepted / args.steps, "p50_ms": statistics.median(step_ms),
                       "p90_ms": sorted(step_ms)[int(0.9 * (len(step_ms) - 1))], "mean_prefix": mean_P,
                       "step_tokens_per_s": wl.M / (ms_per_step * 1e-3)},
        "e2e": None if args.ncu else {
            "value": e2e_tps, "unit": "committed tokens/s (la_generate, prefill included)",
            "h2d_bytes_per_step": gst["h2d_bytes"] / max(gen_steps, 1),
            "d2h_bytes_per_step": gst["d2h_bytes"] / max(gen_steps, 1),
            "bytes_counted_by": "la_stats h2d_bytes / d2h_bytes over the timed la_generate (prompt and initial "
                                "window in; the step state with the accepted tokens out, once per step and once "
                                "for the prefill), divided by its steps",
            "tokens": len(toks), "steps": gen_steps, "seconds": e2e_s},
        "gpu_launches": int(launches),
        "roofline": {"bound": "hbm", "kernel": "k_gemm_tc2 (2-SM tcgen05 projection GEMM, all launches of a step; "
                               "algorithmic bytes = the weights each launch streams)",
                     "achieved": gemm_gbs, "peak": peak, "unit": "GB/s",
                     "frac": (gemm_gbs / peak) if gemm_gbs else None, "traffic": gemm_traffic(),
                     "peak_source": peak_kind, "launch_ms": pst["gemm_ms"] / max(pst["gemm_launches"], 1),
                     "bytes_per_launch": pst["gemm_bytes"] / max(pst["gemm_launches"], 1),
                     "share_of_step": pst["gemm_ms"] / max(pst["steps"], 1) / ms_per_step},
        "step_roofline": {"bytes_per_step": step_bytes, "achieved": step_gbs, "peak": peak, "unit": "GB/s",
                          "frac": step_gbs / peak, "peak_source": peak_kind,
                          "roofline_ms": step_bytes / (peak * 1e9) * 1e3},
        "attention": {"achieved": attn_gbs, "unit": "GB/s",
                      "ms_per_step": pst["attn_ms"] / max(pst["steps"], 1)},
        "breakdown_ms_per_step": {k: pst[k + "_ms"] / max(pst["steps"], 1) for k in ("gemm", "attn", "elem", "spec")},
        "ar_baseline": None if ar_ms is None else {
            "ms_per_token": ar_ms, "tokens_per_s": 1e3 / ar_ms,
            "lookahead_over_ar": (accepted_all / (max_ms * 1e-3)) / (1e3 / ar_ms),
            "note": "la_ar_step (one row per forward, same kernels and weights) timed on this GPU; random weights "
                    "accept A = 1 token per lookahead step, so the ratio is the step cost ratio, not the pages' "
                    "speedup on trained models"},
        "prefill": None if prefill_ms is None else {
            "tokens": len(prompt), "ms": prefill_ms, "tokens_per_s": len(prompt) / (prefill_ms * 1e-3),
            "note": "la_prefill from a host prompt (copy in, 256-row passes through the GEMM and attention kernels, each "
                    "pass streaming every weight once, first token read back); not part of value or ms_per_step"},
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline and not args.ncu and world == 1:
        t1, t0 = oracle_step_sample(weights, wl, prompt, 0)
        step_s = extrapolated_step_seconds(t1, t0, d.n_layers)
        a = accepted / args.steps
        line["cpu_baseline"] = {"value": a / step_s, "unit": "committed tokens/s", "cores": blas_threads(),
                                "kind": "oracle",
                                "sample": "oracle (numpy fp64) forward of one step's M rows through layer 0 with "
                                          "a 256-token prefix, and through embedding+lm_head alone; step time = "
                                          f"{d.n_layers} x layer + head = {step_s:.2f} s; tokens/step taken from "
                                          "the GPU run (same greedy decisions)"}
    dec.close()
    return line


def main():
    args = parse()
    import synth
    wl = synth.WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        # CPU oracle arm: rank 0 alone works and prints; other ranks exit 0.
        if rank == 0:
            print(json.dumps(run_reference(args, wl)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    import synth as _s
    _s.build_generator()
    from exact_decoding_gb300 import build as b
    b.build()
    line = run_ours(args, wl, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
