"""Bench of the MoE-FFN forward layer on B300: tokens/s and grouped-GEMM TFLOPS.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--T TOKENS] [--no-cpu] [--no-e2e] [--e2e-depth D] [--no-extra]
                    [--noise-std S] [--expert-choice] [--backward] [--fp8] [--gemm-one-cta] [--graph]

A step is one whole forward pass of the layer (router with the dispatch scan
in its last CTA, gather, expert GEMM 1, expert GEMM 2, combine) over one batch
of T synthetic tokens.  The step time is taken over K plain calls; K more calls
record the library's stage events for the per-kernel breakdown.  The
default workload is the Mixtral-shaped layer (T=16384, d=4096, f=14336, E=8,
k=2, SwiGLU, bf16) on which the grouped-GEMM bar is stated.  Inputs are larger
than L2 (x is 134 MB, expert weights 2.8 GB), so no L2 flush is done.

The default run also times the four other workloads of the layer (the tiny
fp32 top-1, GPT-2-width top-2 GELU, skewed top-2 with capacity, and
DeepSeek-style fine-grained + shared experts) after the headline, one replica
each, and reports them under other_workloads: tokens/s, per-kernel times and
fractions, and the CUDA-graph replay.  The headline value, roofline and e2e
stay on the Mixtral-shaped layer.  The roofline fraction is taken against the
measured burst bf16 peak: the timed region lasts well under a second.

The end-to-end figure (e2e) calls moe_forward_host on pinned host buffers,
the steps rotating over D streams and workspaces (--e2e-depth, default 3) so
that each step's copies overlap other steps' kernels.

--expert-choice, --fp8 (alone or together) and --backward time those variants
of the step on the same workload; --graph adds the same forward replayed from
a CUDA graph.

Prints one JSON line on rank 0.  Under torchrun each rank runs an independent
replica of the layer on its own GPU (the layer has no cross-GPU step); value is
the total tokens/s of all ranks over the slowest rank's time.

--impl reference times the fp64 CPU oracle on this host's cores instead, on a
bounded sample of the same workload (routing of all T tokens plus the expert
FFNs of a few tokens, extrapolated to T).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import seeded_inputs as si  # noqa: E402

METRIC = "MoE-layer tokens/s on 1 B300; grouped-GEMM TFLOPS as % of bf16 peak"
METRIC_FP8 = "MoE-layer tokens/s on 1 B300 with FP8 (E4M3) experts; grouped-GEMM TFLOPS as % of fp8 peak"
DEFAULT_WORKLOAD = "mixtral_swiglu_bf16"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_desc(cfg):
    act = {si.RELU: "ReLU", si.GELU: "GELU", si.SWIGLU: "SwiGLU"}[cfg.act]
    gate = {si.SOFTMAX: "softmax", si.SIGMOID_NORM: "normalised sigmoid"}[cfg.gating]
    dt = {si.F32: "fp32", si.BF16: "bf16"}[cfg.dtype]
    cap = f", capacity factor {cfg.capacity_factor}" if cfg.capacity_factor > 0 else ""
    sh = f", {cfg.S} shared experts" if cfg.S else ""
    return (f"{cfg.name}: T={cfg.T}, d_model={cfg.d}, d_ff={cfg.f}, E={cfg.E}, k={cfg.k}{sh}, {act} experts, "
            f"{gate} gating, {dt}{cap}")


def algorithmic(cfg, rows_A: int):
    """Per-forward algorithmic work.  rows_A = kept assignments + S * T."""
    T, d, f, E, m = cfg.T, cfg.d, cfg.f, cfg.E, cfg.n_mats
    b = 2 if cfg.dtype == si.BF16 else 4
    g1 = 2.0 * rows_A * d * f * (m - 1)         # x W1 (and x W3)
    g2 = 2.0 * rows_A * f * d                   # h W2
    kept = rows_A - cfg.S * T
    # token choice reads each token's row once and writes it to each kept
    # slot; expert choice reads one x row per grouped row
    gather_read = kept * d * b if getattr(cfg, "expert_choice", False) else T * d * b
    out = {
        "gemm1_flop": g1, "gemm2_flop": g2,
        "router_bytes": T * d * b + d * E * b + T * cfg.k * 8.0,
        "gather_bytes": gather_read + kept * d * b,
        "combine_bytes": rows_A * d * 4.0 + T * d * b,
    }
    if getattr(cfg, "fp8_experts", False):
        # x read in bf16, one E4M3 code per element written per kept slot (and
        # once in token order for the shared experts), one scale per row
        out["gather_bytes"] = T * d * b + kept * (d + 4.0) + (T * (d + 4.0) if cfg.S else 0.0)
        if getattr(cfg, "expert_choice", False):
            # expert choice: x quantised once per token, then each grouped row
            # copies its token's codes and scale
            out["gather_bytes"] = T * d * b + T * (d + 4.0) + 2.0 * kept * (d + 4.0)
        # H read in bf16, codes and one scale per row written
        out["quantize_h_bytes"] = rows_A * (f * 3.0 + 4.0)
    return out


# ---------------------------------------------------------------------------------------------
# ranks: each runs an independent replica of the layer (the layer has no cross-GPU step)


def max_over_ranks(ms: float, device, world: int) -> float:
    """The slowest rank's time: the job's time for a step."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(tokens_per_rank: int, ms_per_step: float, world: int) -> float:
    """Tokens/s of the whole job: every rank's tokens over the slowest rank's step time."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


# ---------------------------------------------------------------------------------------------
# DRAM traffic of the dominant kernel, from the committed ncu summary


GEMM_PAIR_SOURCES = ("grouped_gemm_2sm.cu", "ptx.cuh", "tcgen05.cuh", "common.cuh", "kernels.cuh")


def gemm_source_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in GEMM_PAIR_SOURCES:
        with open(os.path.join(ROOT, "sparse_mixture_experts_48_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(cfg, kernel: str, one_cta: bool):
    """dram read + write bytes per launch of `kernel` from
    profiles/dram_traffic_<workload>.md, if a row matches the workload's T and
    the kernel's sources are unchanged since the capture; else None."""
    path = os.path.join(ROOT, "profiles", f"dram_traffic_{cfg.name}.md")
    if one_cta or not os.path.exists(path):
        return None
    sha = gemm_source_sha()
    for line in open(path, encoding="utf-8"):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 6 and cells[0] == kernel and cells[1] == str(cfg.T) and cells[2] == sha:
            return int(cells[5])
    return None


def measure_fp8_peak(dev, n: int = 8192, reps: int = 10):
    """Dense E4M3 tensor throughput of the vendor library on this GPU: an
    n x n x n cuBLASLt GEMM through torch._scaled_mm (per-tensor scales, bf16
    output), best of `reps` after warm-up, in TFLOP/s.  None if unavailable."""
    import torch
    try:
        a = torch.randn((n, n), device=dev).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), device=dev).to(torch.float8_e4m3fn).t()      # column-major
        one = torch.ones((), device=dev)
        for _ in range(3):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        del a, b
        torch.cuda.empty_cache()
        return 2.0 * n ** 3 / (best / 1e3) / 1e12
    except (RuntimeError, AttributeError, TypeError):
        return None


# ---------------------------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.start = 0

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # the timed region starts once samples flow (nvidia-smi takes a
            # moment to start); only the samples after that are summarised
            t_end = time.time() + 3.0
            while not self.lines and time.time() < t_end and self.proc.poll() is None:
                time.sleep(0.005)
            self.start = len(self.lines)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[self.start:]:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)


def oracle_sample(cfg, inp, n_ffn_tokens: int, seed: int = 0):
    """Time the oracle on all T tokens' routing plus n tokens' expert FFNs;
    return (seconds extrapolated to the full batch, description, seconds the
    sample took)."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    logits = oracle.router_logits(inp["x"], inp["W_g"], inp["b_g"], cfg.dtype)
    r = oracle.routing(cfg, logits)
    t_route = time.perf_counter() - t0
    rows = np.random.default_rng(seed).choice(cfg.T, size=n_ffn_tokens, replace=False)
    t1 = time.perf_counter()
    oracle.layer_rows(cfg, rows, inp, r["topk_idx"], r["topk_w"], r["dropped"])
    t_ffn = time.perf_counter() - t1
    total = t_route + t_ffn * cfg.T / n_ffn_tokens
    desc = (f"routing, dispatch and statistics of all {cfg.T} tokens ({t_route:.2f} s) + expert FFNs and "
            f"combine of {n_ffn_tokens} random tokens ({t_ffn:.2f} s), extrapolated linearly to {cfg.T} tokens")
    return total, desc, t_route + t_ffn


# One oracle sample: the FFNs of as many tokens as take about this long, beside
# the routing of all T tokens.  The reference arm times K + W such samples and
# the CPU baseline CPU_SAMPLES of them, so both legs time the same sample.
SAMPLE_BUDGET_S = 2.0
CPU_SAMPLES = 5


def ffn_sample_size(cfg, budget_s: float = SAMPLE_BUDGET_S) -> int:
    # ~1.5 GMAC/s for the oracle's fp64 loops; per token (k + S) experts of m d f MACs
    per_tok = (cfg.k + cfg.S) * cfg.n_mats * cfg.d * cfg.f / 1.5e9
    return int(max(2, min(cfg.T, budget_s / max(per_tok, 1e-9))))


def run_reference(args, cfg):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = si.layer_inputs(cfg, seed=0)
    n = ffn_sample_size(cfg)
    times, walls, descs = [], [], []
    for i in range(args.warmup + args.steps):
        s, desc, wall = oracle_sample(cfg, inp, n, seed=i)
        if i >= args.warmup:
            times.append(s)
            walls.append(wall)
            descs.append(desc)
    sec = statistics.median(times)
    value = cfg.T / sec
    # A step is one bounded sample (its measured wall time is ms_per_step);
    # value is the full layer's tokens/s extrapolated from it.
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.median(walls) * 1e3,
        "extrapolated_ms_per_full_batch": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "T": cfg.T, "parallelism": "single host thread"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": descs[0] + f"; a step is this sample, value the median over {args.steps} "
                                             f"steps extrapolated to the full batch"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------------
# backward pass


def run_backward(args, cfg, d, dev, world, rank, local):
    """Times moe_backward (the forward recomputed inside, then all gradients) on
    the same workload; prints one JSON line with tokens/s of the training step
    and the GEMM throughput (forward 2 A d f m + backward 2 A d f (2 m - 1))."""
    import torch
    import sparse_mixture_experts_48_b300 as moe
    dy = d["x"].clone()                       # any [T, d] bf16 upstream gradient
    args_in = [d[n] for n in ("x", "W_g", "b_g", "W1", "b1", "W2", "b2", "W3")]
    g = moe.backward(cfg, *args_in, dy)
    ws = g.workspace
    for _ in range(args.warmup):
        moe.backward(cfg, *args_in, dy, workspace=ws)
    if moe.check_device_errors(ws) != 0:
        raise SystemExit("device error in the backward warm-up")
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        e0.record()
        for _ in range(args.steps):
            moe.backward(cfg, *args_in, dy, workspace=ws)
        e1.record()
        torch.cuda.synchronize()
    if moe.check_device_errors(ws) != 0:
        raise SystemExit("device error in the backward timed region")
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev, world)
    fwd = moe.forward(cfg, *args_in)
    torch.cuda.synchronize()
    rows_A = int(fwd.expert_counts.sum().item()) + cfg.S * cfg.T
    m = cfg.n_mats
    flop = 2.0 * rows_A * cfg.d * cfg.f * m + 2.0 * rows_A * cfg.d * cfg.f * (2 * m - 1)
    peaks, kind = load_peaks()
    tf = flop / (ms / 1e3) / 1e12
    sust = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    if rank == 0:
        print(json.dumps({
            "metric": "MoE-layer backward (forward recomputation + gradients) tokens/s on 1 B300",
            "value": replica_throughput(cfg.T, ms, world), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_desc(cfg), "T": cfg.T,
                       "routing": "expert choice" if getattr(cfg, "expert_choice", False) else "token choice"},
            "gemm_flop_per_step": flop, "gemm_tflops": round(tf, 1),
            "frac_of_bf16_sustained": round(tf / sust, 4),
            # the call's GEMM work over the whole call's time: a lower bound of
            # the GEMMs' own rate (their share of the call is about 96 %)
            "roofline": {"bound": "tensor", "kernel": "all expert GEMMs of the call (timed as the whole call)",
                         "achieved": round(tf, 1), "peak": sust, "unit": "TFLOP/s", "frac": round(tf / sust, 4),
                         "traffic": None,
                         "peak_source": f"{kind} bf16_tflops_sustained (cuBLAS bf16, back to back)"},
            "peak_source": kind, "clocks": clocks.summary()}), flush=True)


# ---------------------------------------------------------------------------------------------


# ---------------------------------------------------------------------------------------------
# one workload on the device: the timed loop, per-kernel times and fractions


def measure(cfg, d, args_in, noise, experts8, args, dev, world, peaks, graph=False, barrier=None,
            clock_ctx=None):
    """Times args.steps forward steps after args.warmup warm-ups on device
    buffers, with the library's stage events between its launches (on the
    launching stream).  Returns the step time (max over ranks), per-kernel
    times with their algorithmic GB/s or TFLOP/s and roofline fractions, and
    the graph-replay time when ``graph``."""
    import contextlib
    import torch
    import sparse_mixture_experts_48_b300 as moe
    fp8 = experts8 is not None
    out = moe.alloc_outputs(cfg, dev)
    ws = moe.alloc_workspace(cfg, dev)
    K, W = args.steps, args.warmup
    n_ev = moe.NUM_STAGES + (2 if fp8 else 1)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(K)]
    one_cta = getattr(args, "gemm_one_cta", False)

    def step(i=None):
        if fp8:
            moe.forward_fp8(cfg, d["x"], d["W_g"], d["b_g"], experts8, d["b1"], d["b2"], router_noise=noise,
                            out=out, workspace=ws, stage_events=ev[i] if i is not None else None)
        else:
            moe.forward(cfg, *args_in, router_noise=noise, out=out, workspace=ws,
                        stage_events=ev[i] if i is not None else None, gemm_single_cta=one_cta)

    def sync_all():
        torch.cuda.synchronize()
        if barrier is not None:
            barrier()

    for _ in range(W):
        step()
    status = moe.check_device_errors(ws)
    if status != 0:
        raise SystemExit(f"device error during warm-up: {moe.STATUS.get(status)}")
    sync_all()
    # The step time is taken over K plain calls; the per-kernel breakdown
    # comes from K more calls that record the library's stage events.
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with (clock_ctx if clock_ctx is not None else contextlib.nullcontext()):
        t_start.record()
        for _ in range(K):
            step()
        t_end.record()
        torch.cuda.synchronize()
    if barrier is not None:
        barrier()
    status = moe.check_device_errors(ws)
    if status != 0:
        raise SystemExit(f"device error in the timed region: {moe.STATUS.get(status)}")
    ms_step = max_over_ranks(t_start.elapsed_time(t_end), dev, world) / K

    # The per-kernel breakdown: K more calls that record the stage events,
    # right after the plain calls (so that the plain calls carry none of the
    # events' cost, and the kernels run in the same state of the power cap).
    for i in range(K):
        step(i)
    torch.cuda.synchronize()
    status = moe.check_device_errors(ws)
    if status != 0:
        raise SystemExit(f"device error in the stage-event calls: {moe.STATUS.get(status)}")

    # Last, the same step captured once in a CUDA graph and replayed: no
    # host-side launch work per step (what bounds small layers).
    gres = None
    if graph:
        if fp8:
            fg = moe.ForwardGraph(cfg, d["x"], d["W_g"], d["b_g"], experts=experts8, router_noise=noise)
        else:
            fg = moe.ForwardGraph(cfg, *args_in, router_noise=noise, gemm_single_cta=one_cta)
        for _ in range(W):
            fg.replay()
        sync_all()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record()
        for _ in range(K):
            fg.replay()
        g1.record()
        torch.cuda.synchronize()
        st = moe.check_device_errors(fg.out.workspace)
        if st != 0:
            raise SystemExit(f"device error in the graph loop: {moe.STATUS.get(st)}")
        g_ms = max_over_ranks(g0.elapsed_time(g1) / K, dev, world)
        gres = {"value": replica_throughput(cfg.T, g_ms, world), "unit": "tokens/s", "ms_per_step": g_ms}
        del fg
    # per-kernel durations from the stage events; with FP8 experts event
    # NUM_STAGES + 1 splits GEMM 1 -> GEMM 2 into the H quantisation and GEMM 2
    names = list(moe.STAGE_NAMES)
    spans = [(s, s + 1) for s in range(moe.NUM_STAGES)]
    if fp8:
        g2 = names.index("expert_gemm2")
        q = moe.NUM_STAGES + 1
        spans[g2] = (q, g2 + 1)
        spans.append((g2, q))
        names.append("quantize_h")
    stage_ms = np.array([[ev[i][a].elapsed_time(ev[i][b]) for a, b in spans] for i in range(K)])
    stage_avg = stage_ms.mean(axis=0)
    rows_A = int(out.expert_counts.sum().item()) + cfg.S * cfg.T
    alg = algorithmic(cfg, rows_A)
    hbm = float(peaks["hbm_gbs"])
    tc_burst = float(peaks["bf16_tflops"])
    tc_sust = float(peaks.get("bf16_tflops_sustained", tc_burst))
    tc_tag = "bf16"
    if fp8:
        # E4M3 tensor-core peak: a cuBLASLt E4M3 GEMM measured in this run
        # (peaks["fp8_tflops"]) when there is one, else the measured bf16
        # figures times the nominal dense ratio 4.5 / 2.25 PFLOP/s
        if peaks.get("fp8_tflops"):
            tc_burst = float(peaks["fp8_tflops"])
            tc_sust = tc_burst * (tc_sust / float(peaks["bf16_tflops"]))
        else:
            tc_burst, tc_sust = 2.0 * tc_burst, 2.0 * tc_sust
        tc_tag = "fp8"
    kernels = {name: {"ms": round(float(stage_avg[s]), 5)} for s, name in enumerate(names)}
    hbm_kernels = [("router", "router_bytes"), ("gather", "gather_bytes"), ("combine", "combine_bytes")]
    if fp8:
        hbm_kernels.append(("quantize_h", "quantize_h_bytes"))
    for name, key in hbm_kernels:
        gbs = alg[key] / (stage_avg[names.index(name)] / 1e3) / 1e9
        kernels[name].update({"GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4), "bytes": alg[key]})
    # dispatch as a whole: from the router's end (its last CTA has run the
    # scan) to the gather's end
    disp_ms = stage_avg[names.index("select")] + stage_avg[names.index("gather")]
    gbs = alg["gather_bytes"] / (disp_ms / 1e3) / 1e9
    kernels["dispatch"] = {"ms": round(float(disp_ms), 5), "GB/s": round(gbs, 1),
                           "frac_hbm": round(gbs / hbm, 4), "bytes": alg["gather_bytes"],
                           "spans": "router end to gather end (select + gather stages)"}
    bf16_path = cfg.dtype == si.BF16
    for name, key in (("expert_gemm1", "gemm1_flop"), ("expert_gemm2", "gemm2_flop")):
        tf = alg[key] / (stage_avg[names.index(name)] / 1e3) / 1e12
        kernels[name].update({"TFLOP/s": round(tf, 1), "flop": alg[key]})
        if bf16_path:
            kernels[name].update({f"frac_{tc_tag}_burst": round(tf / tc_burst, 4),
                                  f"frac_{tc_tag}_sustained": round(tf / tc_sust, 4)})
    gemm_ms = stage_avg[names.index("expert_gemm1")] + stage_avg[names.index("expert_gemm2")]
    if fp8:
        gemm_ms += stage_avg[names.index("quantize_h")]
    gemm_tf = (alg["gemm1_flop"] + alg["gemm2_flop"]) / (gemm_ms / 1e3) / 1e12
    grouped = {"tflops": round(gemm_tf, 1), "ms": round(float(gemm_ms), 4)}
    if bf16_path:
        grouped.update({f"frac_of_{tc_tag}_burst": round(gemm_tf / tc_burst, 4),
                        f"frac_of_{tc_tag}_sustained": round(gemm_tf / tc_sust, 4)})

    return {"out": out, "ws": ws, "ms_step": ms_step, "kernels": kernels, "grouped_gemm": grouped,
            "graph": gres, "tc_burst": tc_burst, "tc_sust": tc_sust, "rows_A": rows_A,
            # router (with the dispatch scan in its last CTA), gather, GEMM 1,
            # GEMM 2, combine; + the H quantisation with FP8 experts; + the
            # per-expert selection with expert choice (+ x's quantisation per
            # token with both)
            "launches_per_step": 5 + (1 if fp8 else 0) + (1 if getattr(cfg, "expert_choice", False) else 0)
            + (1 if fp8 and getattr(cfg, "expert_choice", False) else 0)}


def other_configs(args, dev, peaks):
    """The other workloads of the layer in the same run (one replica): per
    workload tokens/s, per-kernel times and fractions, and the CUDA-graph
    replay (what bounds the small, launch-bound layers)."""
    import torch
    res = {}
    for name in si.CONFIG_ORDER:
        if name == DEFAULT_WORKLOAD:
            continue
        cfg = si.CONFIGS[name]
        inp = si.layer_inputs(cfg, seed=0)

        def to_dev(a):
            if a is None:
                return None
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
            return torch.from_numpy(a).to(dev)

        d = {k: to_dev(v) for k, v in inp.items()}
        args_in = [d[n] for n in ("x", "W_g", "b_g", "W1", "b1", "W2", "b2", "W3")]
        r = measure(cfg, d, args_in, None, None, args, dev, 1, peaks, graph=True)
        res[name] = {"workload": workload_desc(cfg), "value": cfg.T / (r["ms_step"] / 1e3), "unit": "tokens/s",
                     "ms_per_step": r["ms_step"], "graph": r["graph"], "grouped_gemm": r["grouped_gemm"],
                     "kernels": r["kernels"], "rows_A": r["rows_A"],
                     "l2": "x %.1f MB, expert weights %.1f MB" % (
                         inp["x"].nbytes / 1e6, sum(inp[n].nbytes for n in ("W1", "W2", "W3")
                                                    if inp[n] is not None) / 1e6)}
        del d, args_in, r
        torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=si.CONFIG_ORDER)
    ap.add_argument("--T", type=int, default=0, help="override the token count (profiling runs)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end loop")
    ap.add_argument("--e2e-depth", type=int, default=3,
                    help="streams (and workspaces) the end-to-end loop rotates over (>= 2; 3 measured best: "
                         "a stream's copies out and in then have two other steps' kernels to hide behind)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads (reported under other_workloads by the default run)")
    ap.add_argument("--noise-std", type=float, default=0.0,
                    help="add seeded Gaussian router noise of this std before gating and top-k (0: none)")
    ap.add_argument("--expert-choice", action="store_true",
                    help="expert-choice routing: each expert takes its C = ceil(T k / E) best tokens")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (moe_backward: forward recomputation + gradients) instead")
    ap.add_argument("--gemm-one-cta", action="store_true",
                    help="bf16 expert GEMMs on the one-CTA tile kernel instead of the CTA-pair kernel")
    ap.add_argument("--graph", action="store_true",
                    help="also time the layer captured in a CUDA graph and replayed (reported under 'graph')")
    ap.add_argument("--fp8", action="store_true",
                    help="FP8 (E4M3) expert weights and activations (moe_forward_fp8); the weights are "
                         "quantised once before the timed region")
    args = ap.parse_args()
    cfg = si.CONFIGS[args.workload]
    if args.T:
        cfg = cfg.replace(T=args.T)
    if args.expert_choice:
        cfg = cfg.replace(expert_choice=True)
    if args.fp8:
        if args.backward or args.gemm_one_cta or args.impl == "reference":
            raise SystemExit("--fp8 runs the forward on the CTA-pair GEMM of our implementation")
        cfg = cfg.replace(fp8_experts=True)
        args.no_cpu = True
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)

    if args.impl == "reference":
        return run_reference(args, cfg)

    import torch
    import torch.distributed as dist

    import sparse_mixture_experts_48_b300 as moe
    from sparse_mixture_experts_48_b300 import build as mbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if rank == 0:
        mbuild.build()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        dist.barrier()
        mbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    inp = si.layer_inputs(cfg, seed=rank)

    def to_dev(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    d = {k: to_dev(v) for k, v in inp.items()}
    args_in = [d[n] for n in ("x", "W_g", "b_g", "W1", "b1", "W2", "b2", "W3")]
    noise = to_dev(si.router_noise(cfg, seed=rank, std=args.noise_std)) if args.noise_std > 0 else None
    if args.backward:
        return run_backward(args, cfg, d, dev, world, rank, local)
    experts8 = moe.quantize_experts_fp8(d["W1"], d["W2"], d["W3"]) if args.fp8 else None
    if args.fp8:
        # the layer keeps only the E4M3 codes and scales of the expert weights
        torch.cuda.synchronize()
        for n in ("W1", "W2", "W3"):
            d[n] = None
        args_in = None
        torch.cuda.empty_cache()
    peaks, peak_kind = load_peaks()
    if args.fp8:
        fp8_peak = measure_fp8_peak(dev)
        if fp8_peak:
            peaks = dict(peaks, fp8_tflops=fp8_peak)
    K, W = args.steps, args.warmup

    def barrier():
        if world > 1:
            dist.barrier()

    clocks = ClockSampler(local)
    res = measure(cfg, d, args_in, noise, experts8, args, dev, world, peaks, graph=args.graph,
                  barrier=(dist.barrier if world > 1 else None), clock_ctx=clocks)
    out = res["out"]
    ms_step = res["ms_step"]
    value = replica_throughput(cfg.T, ms_step, world)
    kernels = res["kernels"]
    fp8 = args.fp8
    dom = "expert_gemm1"
    tc_tag = "fp8" if fp8 else "bf16"
    dom_tf = kernels[dom]["TFLOP/s"]
    tc_burst, tc_sust = res["tc_burst"], res["tc_sust"]
    traffic = measured_traffic(cfg, dom + ("_fp8" if fp8 else ""), args.gemm_one_cta)
    if fp8 and peaks.get("fp8_tflops"):
        src = ("cuBLASLt E4M3 GEMM 8192^3 (torch._scaled_mm, per-tensor scales, bf16 out) measured in this run: "
               "best of 10, burst")
    elif fp8:
        src = "measured bf16_tflops x 2 (burst; nominal E4M3 / bf16 dense ratio)"
    else:
        src = "measured bf16_tflops (cuBLAS bf16 burst: the timed region is well under a second)"
    if peak_kind != "measured":
        src = src.replace("measured", "fallback")
    roofline = {"bound": "tensor", "kernel": dom, "achieved": dom_tf, "peak": tc_burst, "unit": "TFLOP/s",
                "frac": round(dom_tf / tc_burst, 4), "traffic": traffic, "peak_source": src,
                "frac_of_sustained_peak": round(dom_tf / tc_sust, 4),
                "timed_region_s": round(ms_step * args.steps / 1e3, 3)}
    graph = res["graph"]
    grouped = res["grouped_gemm"]

    # End to end through the public API with host buffers (moe_forward_host):
    # every step copies its x from page-locked host memory in and all outputs
    # back out.  Steps rotate over D streams and D workspaces (D =
    # --e2e-depth), so a step's copies overlap the other steps' kernels; the
    # timed region spans all K steps.
    e2e = None
    if not args.no_e2e:
        x_host = torch.empty(d["x"].shape, dtype=d["x"].dtype, pin_memory=True)
        x_host.copy_(d["x"].cpu())
        noise_host = noise.cpu().pin_memory() if noise is not None else None
        weights = args_in[1:] if args_in is not None else None
        D = max(2, args.e2e_depth)
        streams = [torch.cuda.Stream(device=dev) for _ in range(D)]
        hws = [torch.empty((moe.host_workspace_size(cfg),), dtype=torch.uint8, device=dev) for _ in range(D)]
        houts = [moe.alloc_host_outputs(cfg) for _ in range(D)]

        def e2e_step(i):
            if fp8:
                moe.forward_fp8_host(cfg, x_host, d["W_g"], d["b_g"], experts8, d["b1"], d["b2"],
                                     router_noise_host=noise_host, out=houts[i % D], workspace=hws[i % D],
                                     stream=streams[i % D])
            else:
                moe.forward_host(cfg, x_host, *weights, router_noise_host=noise_host, out=houts[i % D],
                                 workspace=hws[i % D], stream=streams[i % D], gemm_single_cta=args.gemm_one_cta)

        for i in range(W):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(streams[0])
        for st_ in streams[1:]:
            st_.wait_event(e0)
        for i in range(K):
            e2e_step(i)
        for st_ in streams[1:]:
            last = torch.cuda.Event()
            last.record(st_)
            streams[0].wait_event(last)
        e1.record(streams[0])
        torch.cuda.synchronize()
        barrier()
        for hw in hws:
            st = moe.check_device_errors(hw)
            if st != 0:
                raise SystemExit(f"device error in the end-to-end loop: {moe.STATUS.get(st)}")
        e_ms = e0.elapsed_time(e1) / K
        e_ms = max_over_ranks(e_ms, dev, world)
        ho = houts[0]
        bi = x_host.numel() * x_host.element_size() + (noise_host.numel() * 4 if noise_host is not None else 0)
        bo = sum(t.numel() * t.element_size() for t in (ho.y, ho.topk_idx, ho.topk_w, ho.expert_counts,
                                                         ho.dropped_mask, ho.f, ho.P, ho.L_aux))
        e2e = {"value": replica_throughput(cfg.T, e_ms, world), "unit": "tokens/s", "ms_per_step": e_ms,
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "how": ("moe_forward_fp8_host" if fp8 else "moe_forward_host") +
                      f", pinned host x in / all outputs out every step, {D} streams x {D} workspaces"}

    cpu = None
    if rank == 0 and not args.no_cpu:
        n = ffn_sample_size(cfg)
        runs = [oracle_sample(cfg, inp, n, seed=i) for i in range(CPU_SAMPLES)]
        sec = statistics.median(r[0] for r in runs)
        cpu = {"value": cfg.T / sec, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": runs[0][1] + f"; median of {CPU_SAMPLES} such samples "
                                      f"({sum(r[2] for r in runs):.1f} s of CPU work); single thread of "
                                      f"{os.cpu_count()} host cores"}

    # The other workloads, on rank 0, after the headline's timed region: the
    # default run reports every workload of the layer.
    others = None
    if (rank == 0 and not args.no_extra and args.workload == DEFAULT_WORKLOAD and not args.T and not fp8
            and not args.expert_choice and not args.gemm_one_cta and args.noise_std == 0):
        others = other_configs(args, dev, peaks)

    if rank == 0:
        line = {
            "metric": METRIC_FP8 if fp8 else METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": W,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3" if fp8 else ("bf16" if cfg.dtype == si.BF16 else "f32"), "data": "synthetic",
            "config": {"workload": workload_desc(cfg), "T": cfg.T, "d_model": cfg.d, "d_ff": cfg.f, "E": cfg.E,
                       "k": cfg.k, "n_shared": cfg.S, "parallelism": "replicas" if world > 1 else "single GPU",
                       "expert_gemm": "one-CTA 128x256 tiles" if args.gemm_one_cta else "CTA-pair 256x256 tiles",
                       "router_noise_std": args.noise_std,
                       "routing": "expert choice" if args.expert_choice else "token choice",
                       "experts": ("FP8 E4M3 weights (one scale per output unit) and activations (one scale "
                                   "per row); router, x, y in bf16" if fp8 else "bf16"),
                       "l2": "no flush: inputs larger than L2 (x %.0f MB, expert weights %.2f GB)" % (
                           inp["x"].nbytes / 1e6, sum(inp[n].nbytes for n in ("W1", "W2", "W3")
                                                      if inp[n] is not None) / (2e9 if fp8 else 1e9))},
            "grouped_gemm": grouped,
            "roofline": roofline,
            "kernels": kernels,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "graph": graph,
            "other_workloads": others,
            "gpu_launches": res["launches_per_step"] * K,
            "clocks": clocks.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
