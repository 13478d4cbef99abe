#!/usr/bin/env python
"""Benchmark of the MoE FFN layer, forward + backward, on one GB300 per process.

One step = moe_layer_fwd + moe_layer_bwd over one batch of the workload (default: the
Mixtral-like layer, T = 8192 tokens = 2 x 4096, d_model 4096, 8 experts top-2, d_ff 14336,
dropless), with seeded synthetic inputs and random-init weights of that shape resident in HBM.

Prints one JSON line (rank 0):
  value      tokens/s over all ranks (each rank runs an independent replica: the layer is
             single-GPU by design, so N > 1 is replicas only, weak scaling)
  e2e        the same through the C ABI with the step's inputs (x, dy) copied host->device from
             pinned memory and its results (y, dx) copied back, inside the timed region
  roofline   the dominant kernel: algorithmic work per launch / its CUDA-event duration, against the
             measured peak (MEASURED_PEAKS.json)
  cpu_baseline  the fp64 oracle on a bounded token sample, on this host's cores (rank 0, N = 1)
  workloads  (default Mixtral-like run) a compact record of each other workload -- tiny, DeepSeek-,
             Qwen3- and GPT-OSS-like -- measured the same way over --workload-steps steps, and of
             the Mixtral-, DeepSeek- and Qwen3-like layers with gather_in_gemm = 1 ("+gather_in_gemm")

--impl reference times the oracle alone (on the host cores) on the same workload and metric.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s fwd+bwd"
DESCR = {
    "tiny": "tiny MoE layer: T=256, d=128, E=8 top-2, d_ff=256, SwiGLU, dropless",
    "mixtral": "Mixtral-like MoE layer: T=8192 (2x4096), d=4096, E=8 top-2, d_ff=14336, SwiGLU, dropless",
    "deepseek": "DeepSeek-like MoE layer: T=16384, d=2048, E=64 top-6 renormalised + 2 shared, d_ff=1408",
    "qwen3": "Qwen3-like MoE layer: T=32768, d=2048, E=128 top-8, d_ff=768, Zipf(1.2)-biased router",
    "gptoss": "GPT-OSS-like MoE layer: T=65536 (2x32768), d=2880, E=128 top-4, d_ff=2880, capacity 1.25",
}
GEMMS = {  # algorithmic FLOPs per launch in units of N*d*f (N = rows the experts see, no pads)
    "gemm_gate_up_swiglu": 4, "gemm_down": 2, "gemm_bwd_dgrad_down": 2, "gemm_bwd_recompute_swiglu": 4,
    "gemm_wgrad": 6, "gemm_dgrad_x": 4,
}
HBM_KERNELS = ("dispatch_gather", "combine", "combine_bwd")
ROUTER_KERNELS = ("route_fwd", "router_dlogits")   # the logit pass over x; dl from the kept logits
KERNEL_SOURCES = ("gemm.cu", "dispatch.cu", "combine.cu", "route.cu", "route_tc.cu", "activations.cu", "ptx.cuh",
                  "common.cuh", "tmap.cuh", "e4m3.cuh")
ROW_TILE = 256   # expert segments are padded to multiples of this many rows (include/moe.h)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixtral", choices=list(synth.CONFIGS))
    ap.add_argument("--cpu-tokens", type=int, default=16, help="oracle sample size (tokens)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override T (a smaller case of the same layer shape, for profiler captures)")
    ap.add_argument("--experts", type=int, default=0, help="override E (profiler captures)")
    ap.add_argument("--topk", type=int, default=0, help="override k (profiler captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fp8", action="store_true",
                    help="also time the layer with e4m3 expert GEMMs (forward, and forward + backward) beside bf16")
    ap.add_argument("--keep-rows", type=int, default=0,
                    help="expert-ordered rows whose gate/up pre-activations the forward keeps instead "
                         "of the backward recomputing them (0: recompute all, the default; -1: keep all)")
    ap.add_argument("--keep-budget", type=float, default=None,
                    help="bytes of kept activations (a, b) the layer may hold between forward and backward; "
                         "the library chooses keep_rows from it (moe_keep_rows_for_budget)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="measure the chosen workload only (by default the Mixtral-like line also carries a "
                         "compact record of every other workload)")
    ap.add_argument("--workload-steps", type=int, default=10, help="timed steps of each extra workload")
    ap.add_argument("--gather-in-gemm", action="store_true",
                    help="the expert GEMMs gather x and dy rows from token order (gather_in_gemm = 1) instead of "
                         "reading x_perm / dY_perm written by the dispatch gather")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return {"hbm": p["hbm_gbs"], "tensor": p["bf16_tflops_sustained"], "tensor_burst": p["bf16_tflops"],
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm": 6800.0, "tensor": 1700.0, "tensor_burst": 1900.0, "source": "fallback"}


def fp8_forward(args, mc, cfg, x, W_r, b_r, Wg, Wu, Wd, dy, buf, N, tensor_peak, tensor_kind, pk, ms_bf16_step):
    """The layer with e4m3 expert GEMMs against bf16 on the same inputs, each timed alone over
    args.steps calls with CUDA events: the forward (moe_layer_fwd_fp8 against moe_layer_fwd) and
    the whole step (moe_layer_fwd_fp8 + moe_layer_bwd_fp8 against the bf16 step measured above).
    The weights are quantised once, untimed: row codes of W_gate, W_up, W_down for the forward,
    column codes of W_down and of W_gate over W_up for the backward."""
    import torch
    import mixture_experts_layer_10_gb300 as moe
    T, d, f = cfg["T"], cfg["d"], cfg["f"]
    G = cfg["E"] + cfg["S"]

    def quant(t):
        codes = torch.empty(t.shape, dtype=torch.uint8, device="cuda")
        scales = torch.empty(G, t.shape[1], dtype=torch.float32, device="cuda")
        moe.moe_quantize_rows_e4m3(t, codes, scales)
        return codes, scales
    g8, u8, d8 = quant(Wg), quant(Wu), quant(Wd)
    wdt = (torch.empty(G, f, d, dtype=torch.uint8, device="cuda"), torch.empty(G, f, dtype=torch.float32, device="cuda"))
    moe.moe_quantize_cols_e4m3(Wd, None, *wdt)
    wgut = (torch.empty(G, d, 2 * f, dtype=torch.uint8, device="cuda"),
            torch.empty(G, d, dtype=torch.float32, device="cuda"))
    moe.moe_quantize_cols_e4m3(Wg, Wu, *wgut)
    # without kept activations: the FP8 calls recompute every row from the codes
    mc = moe.config_from(dict(cfg, keep_rows=0))
    y8 = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    dx8 = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    dW_r = torch.empty(d, cfg["E"], dtype=torch.float32, device="cuda")
    db_r = torch.empty(cfg["E"], dtype=torch.float32, device="cuda") if b_r is not None else None
    dWg, dWu, dWd = torch.empty_like(Wg), torch.empty_like(Wu), torch.empty_like(Wd)
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn, profile):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        moe.moe_profile_enable(profile)
        ev0.record(stream)
        for _ in range(args.steps):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize()
        prof = moe.moe_profile_read() if profile else {}
        moe.moe_profile_enable(False)
        status = moe.moe_check_error(buf.ws)
        if status != 0:
            raise RuntimeError(f"fp8 layer failed: {moe.moe_status_string(status)}")
        return ev0.elapsed_time(ev1) / args.steps, prof

    def fwd8():
        moe.moe_layer_fwd_fp8(mc, x, W_r, b_r, *g8, *u8, *d8, y8, buf.saved, buf.ws)

    def step8():
        fwd8()
        moe.moe_layer_bwd_fp8(mc, x, W_r, b_r, *g8, *u8, *wdt, *wgut, buf.saved, dy, dx8, dW_r, db_r, dWg, dWu,
                              dWd, buf.ws)

    ms16, _ = timed(lambda: moe.moe_layer_fwd(mc, x, W_r, b_r, Wg, Wu, Wd, y8, buf.saved, buf.ws), False)
    ms8, prof = timed(fwd8, True)
    ms8_step, prof_step = timed(step8, True)
    peak8 = 2 * tensor_peak
    kern = {}
    for name, flops in (("gemm_gate_up_fp8", 4 * N * d * f), ("gemm_down_fp8", 2 * N * d * f)):
        tot, n = prof.get(name, (0.0, 0))
        if n:
            tf = flops * n / (tot / 1000.0) / 1e12
            kern[name] = {"ms_per_step": tot / args.steps, "tflops": tf, "frac": tf / peak8}
    tot, n = prof.get("quantize_e4m3", (0.0, 0))
    if n:   # the T token rows of x and the N rows of h: bf16 in, codes and a scale out
        gbs = ((T * d + N * f) * 3 + 4 * (T + N)) * args.steps / (tot / 1000.0) / 1e9
        kern["quantize_e4m3"] = {"ms_per_step": tot / args.steps, "gbs": gbs, "frac": gbs / pk["hbm"]}
    step_kern = {}
    for name, flops in (("gemm_bwd_dgrad_down_fp8", 2 * N * d * f), ("gemm_bwd_recompute_swiglu_fp8", 4 * N * d * f),
                        ("gemm_dgrad_x_fp8", 4 * N * d * f)):
        tot, n = prof_step.get(name, (0.0, 0))
        if n:
            tf = flops * n / (tot / 1000.0) / 1e12
            step_kern[name] = {"ms_per_step": tot / args.steps, "tflops": tf, "frac": tf / peak8}
    for name in ("gemm_wgrad", "quantize_e4m3", "dispatch_gather", "combine_bwd"):
        tot, n = prof_step.get(name, (0.0, 0))
        if n:
            step_kern[name] = {"ms_per_step": tot / args.steps, "launches": n}
    # the resource model's roofline for both forwards, on the same peaks
    from mixture_experts_layer_10_gb300 import resource_model
    n_routed = N - cfg["S"] * T
    p16 = resource_model.predict_forward_ms(cfg, pk["tensor_burst"], pk["hbm"], N=n_routed)["step_ms"]
    p8 = resource_model.predict_forward_ms(cfg, pk["tensor_burst"], pk["hbm"], N=n_routed, fp8=True)["step_ms"]
    return {"metric": "forward tokens/s (e4m3 expert GEMMs)", "value": T / (ms8 / 1000.0), "fwd_ms": ms8,
            "bf16_fwd_ms": ms16, "speedup_vs_bf16_fwd": ms16 / ms8,
            "step": {"metric": METRIC + " (e4m3 expert GEMMs)", "value": T / (ms8_step / 1000.0),
                     "ms_per_step": ms8_step, "bf16_ms_per_step": ms_bf16_step,
                     "speedup_vs_bf16_step": ms_bf16_step / ms8_step, "kernels": step_kern},
            "model": {"fp8_fwd_predicted_ms": p8, "fp8_measured_over_predicted": ms8 / p8,
                      "bf16_fwd_predicted_ms": p16, "bf16_measured_over_predicted": ms16 / p16},
            "peak_tflops": peak8, "peak_kind": "2 x " + tensor_kind.split(":")[0] + " (nominal fp8:bf16 ratio)",
            "kernels": kern}


def code_only(src: str) -> str:
    """CUDA/C++ source without comments and whitespace runs: what the compiler sees of it."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_source_hash() -> str:
    """Identifies the kernels' code (comments and layout ignored), so recorded counters stay valid
    across comment-only edits and lapse with any code change."""
    h = hashlib.sha256()
    for n in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "mixture_experts_layer_10_gb300", "csrc", n), encoding="utf-8") as fh:
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on today's sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            t = json.load(fh)
        e = t[workload][kernel]
        if e.get("source_hash") != kernel_source_hash():
            return None
        return e["dram_bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms; summary() keeps the samples
    taken between mark_start() and mark_end() (the timed region)."""
    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        self.t0 = self.t1 = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        self.file.flush()
        rows = []
        with open(self.file.name) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        def when(v):
            try:
                return datetime.datetime.strptime(v, "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                return None
        if self.t0 is not None and self.t1 is not None:
            inside = [r for r in rows if when(r[0]) is not None and self.t0 <= when(r[0]) <= self.t1]
            if inside:
                rows = inside
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(rows[0][2]),
                "reasons": reasons, "samples": len(rows),
                "sm_mhz_min": min(sm) if sm else None,
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


def max_over_ranks(value: float, world: int) -> float:
    """The largest of every rank's value (the slowest replica sets the step time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_sample(inp, cfg, n_tokens, seed=1):
    """The oracle as it stands on a seeded sample of tokens: routing, expert forward and
    backward (weight-gradient products included) and the router backward of those tokens."""
    import oracle
    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(cfg["T"], size=min(n_tokens, cfg["T"]), replace=False))
    L = oracle.Layer(inp, cfg)
    t0 = time.perf_counter()
    L.token_outputs(toks)
    return len(toks), time.perf_counter() - t0


def reference_arm(args, rank, world):
    if rank != 0:
        return
    cfg = synth.CONFIGS[args.workload]
    inp = synth.make_inputs(cfg, seed=0)
    times = []
    n = 0
    for i in range(args.warmup + args.steps):
        n, dt = oracle_sample(inp, cfg, args.cpu_tokens, seed=1 + i)
        if i >= args.warmup:
            times.append(dt)
    ms = 1000.0 * sum(times) / len(times)
    value = n / (ms / 1000.0)
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": DESCR[args.workload], "sample_tokens_per_step": n},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} seeded tokens of the {args.workload} workload per step "
                                   f"(fwd + bwd incl. weight-gradient products), numpy/OpenBLAS threads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def device_experts(cfg, seed=0):
    """W_gate, W_up ~ N(0, 1/d) and W_down ~ N(0, 1/d_ff) in bf16, drawn on the device from a seeded
    generator (the extra workloads of the bench line: the routing, which sets every kernel's work,
    still comes from the seeded x, W_r and bias of synth; drawing billions of weights on the host
    would take longer than measuring them)."""
    import torch
    T, d, f, G = cfg["T"], cfg["d"], cfg["f"], cfg["E"] + cfg["S"]
    g = torch.Generator(device="cuda").manual_seed(1000 + seed)
    out = []
    for shape, std in (((G, f, d), d ** -0.5), ((G, f, d), d ** -0.5), ((G, d, f), f ** -0.5)):
        w = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        for e in range(G):
            w[e] = (torch.randn(shape[1:], generator=g, device="cuda") * std).to(torch.bfloat16)
        out.append(w)
    return out


def run_workload(args, name, cfg, steps, warmup, rank, world, local, barrier, extra=False):
    """One workload's measurement: device-resident steps (CUDA events, per-kernel profile, clocks),
    end to end through host buffers, and CUDA-graph replay.  Returns the JSON record."""
    import torch
    import mixture_experts_layer_10_gb300 as moe

    T, d, f, E, k, S = cfg["T"], cfg["d"], cfg["f"], cfg["E"], cfg["k"], cfg["S"]
    G = E + S
    inp = synth.make_inputs(cfg, seed=0, parts=("x", "router", "dy") if extra else ("x", "router", "experts", "dy"))

    def dev_bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    x, dy = dev_bf16(inp["x"]), dev_bf16(inp["dy"])
    W_r = torch.from_numpy(inp["W_r"]).cuda()
    b_r = torch.from_numpy(inp["b_r"]).cuda() if inp["b_r"] is not None else None
    if extra:
        Wg, Wu, Wd = device_experts(cfg)
    else:
        Wg, Wu, Wd = dev_bf16(inp["W_gate"]), dev_bf16(inp["W_up"]), dev_bf16(inp["W_down"])
    mc = moe.config_from(cfg)
    keep_budget = None
    if not extra and args.keep_budget is not None:
        keep_budget = int(args.keep_budget)
        cfg["keep_rows"], _ = moe.moe_keep_rows_for_budget(mc, keep_budget)
        mc = moe.config_from(cfg)
    elif not extra and args.keep_rows:
        cfg["keep_rows"] = moe.moe_perm_rows(mc) if args.keep_rows < 0 else args.keep_rows
        mc = moe.config_from(cfg)
    keep = min(cfg.get("keep_rows", 0) // ROW_TILE * ROW_TILE, moe.moe_perm_rows(mc))
    buf = moe.Buffers.allocate(mc)
    y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    dx = torch.empty_like(y)
    dW_r = torch.empty(d, E, dtype=torch.float32, device="cuda")
    db_r = torch.empty(E, dtype=torch.float32, device="cuda") if b_r is not None else None
    dWg, dWu, dWd = torch.empty_like(Wg), torch.empty_like(Wu), torch.empty_like(Wd)

    def step(xx=x, dyy=dy, yy=y, dxx=dx):
        moe.moe_layer_fwd(mc, xx, W_r, b_r, Wg, Wu, Wd, yy, buf.saved, buf.ws)
        moe.moe_layer_bwd(mc, xx, W_r, b_r, Wg, Wu, Wd, buf.saved, dyy, dxx, dW_r, db_r, dWg, dWu, dWd, buf.ws)

    # rows the experts see (no pads): kept routed slots + shared tokens, from one dispatch
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    gates = torch.empty(T, k, dtype=torch.float32, device="cuda")
    moe.moe_route(mc, x, W_r, b_r, idx, gates, None, buf.ws)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    scratch_rows = torch.empty(T * k, dtype=torch.int32, device="cuda")
    scratch_tok = torch.empty(T * k, dtype=torch.int32, device="cuda")
    x_perm = torch.empty(buf.rows, d, dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch(mc, idx, x, counts, offsets, scratch_rows, scratch_tok, x_perm, buf.ws)
    status = moe.moe_check_error(buf.ws)
    if status != 0:
        raise RuntimeError(f"dispatch failed: {moe.moe_status_string(status)}")
    counts_h = counts.cpu().numpy()
    n_kept = int(offsets[-1].item())
    N = n_kept + S * T
    # rows whose a, b the forward keeps (real rows below `keep` in the padded expert order); the
    # recompute GEMM does the rest
    seg_rows = list(np.diff(offsets.cpu().numpy())) + [T] * S
    start, kept_real = 0, 0
    for n_g in seg_rows:
        kept_real += max(0, min(start + int(n_g), keep) - start)
        start += (int(n_g) + ROW_TILE - 1) // ROW_TILE * ROW_TILE
    load_max_over_mean = float(counts_h.max() / counts_h.mean())
    del x_perm, scratch_rows, scratch_tok

    for _ in range(warmup):
        step()
    status = moe.moe_check_error(buf.ws)
    if status != 0:
        raise RuntimeError(f"layer failed: {moe.moe_status_string(status)}")

    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        moe.moe_profile_enable(True)
        clocks.mark_start()
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        clocks.mark_end()
        barrier()
    prof = moe.moe_profile_read()
    sm_in = moe.moe_profile_sm_clock()   # the SM clock each GEMM kernel ran at (in-kernel cycles / ns)
    moe.moe_profile_enable(False)
    clk = clocks.summary()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / steps, world)
    status = moe.moe_check_error(buf.ws)
    if status != 0:
        raise RuntimeError(f"layer failed in the timed region: {moe.moe_status_string(status)}")

    # End to end through the C ABI with host buffers: every step copies its inputs (x, dy) from
    # pinned host memory and its results (y, dx) back.  A copy stream overlaps step i's compute
    # with step i+1's H2D and step i-1's D2H (double-buffered device inputs and outputs).  Compute
    # runs on a stream of its own: work on the legacy default stream would serialise with every
    # other blocking stream, the copy stream included.
    cstream = torch.cuda.Stream()
    # every host buffer pinned (empty_like does not carry pinning over): a copy to or from pageable
    # memory blocks the host until it completes, which would serialise the next step's launches
    def pinned():
        return torch.empty(T, d, dtype=torch.bfloat16, pin_memory=True)
    x_h, dy_h, y_h, dx_h = pinned().copy_(x.cpu()), pinned().copy_(dy.cpu()), pinned(), pinned()
    assert all(t.is_pinned() for t in (x_h, dy_h, y_h, dx_h))
    xin = [torch.empty_like(x), torch.empty_like(x)]
    dyin = [torch.empty_like(dy), torch.empty_like(dy)]
    yout = [torch.empty_like(y), torch.empty_like(y)]
    dxout = [torch.empty_like(dx), torch.empty_like(dx)]
    copy_stream = torch.cuda.Stream()
    loaded = [torch.cuda.Event(), torch.cuda.Event()]
    computed = [torch.cuda.Event(), torch.cuda.Event()]

    def e2e_run(n):
        copy_stream.wait_stream(cstream)       # the first copy starts inside the timed region
        with torch.cuda.stream(copy_stream):
            xin[0].copy_(x_h, non_blocking=True)
            dyin[0].copy_(dy_h, non_blocking=True)
            loaded[0].record(copy_stream)
        for i in range(n):
            b = i % 2
            cstream.wait_event(loaded[b])
            with torch.cuda.stream(cstream):
                step(xin[b], dyin[b], yout[b], dxout[b])
            computed[b].record(cstream)
            with torch.cuda.stream(copy_stream):
                if i + 1 < n:
                    if i >= 1:
                        copy_stream.wait_event(computed[1 - b])   # step i-1 is done with that buffer
                    xin[1 - b].copy_(x_h, non_blocking=True)
                    dyin[1 - b].copy_(dy_h, non_blocking=True)
                    loaded[1 - b].record(copy_stream)
                copy_stream.wait_event(computed[b])
                y_h.copy_(yout[b], non_blocking=True)
                dx_h.copy_(dxout[b], non_blocking=True)
        cstream.wait_stream(copy_stream)

    cstream.wait_stream(stream)
    e2e_run(2)
    barrier()
    torch.cuda.synchronize()
    ev0.record(cstream)
    e2e_run(steps)
    ev1.record(cstream)
    torch.cuda.synchronize()
    barrier()
    ms_e2e = max_over_ranks(ev0.elapsed_time(ev1) / steps, world)

    # The same device-resident step captured once in a CUDA graph and replayed (launch overhead
    # removed); reported beside the primary, stream-launched number.
    graph = {"ms_per_step": None}
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        with torch.cuda.graph(g):
            step()
        g.replay()
        torch.cuda.synchronize()
        barrier()
        ev0.record(stream)
        for _ in range(steps):
            g.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms_graph = max_over_ranks(ev0.elapsed_time(ev1) / steps, world)
        graph = {"ms_per_step": ms_graph, "value": world * T / (ms_graph / 1000.0), "unit": "tokens/s"}
        del g
    except RuntimeError as err:   # capture unsupported here: say why, keep the stream numbers
        graph = {"ms_per_step": None, "note": str(err).splitlines()[0][:200]}
    status = moe.moe_check_error(buf.ws)
    if status != 0:
        raise RuntimeError(f"layer failed in the graph replays: {moe.moe_status_string(status)}")

    pk = peaks()
    # Denominator for the tensor-bound kernels: the burst cuBLAS figure when the SM clock held at its
    # maximum (as during the burst measurement), else the sustained one (the power cap lowered it, as
    # in the sustained cuBLAS loop).  The clock is the one the GEMM kernels ran at -- their CTAs' SM
    # cycles over nanoseconds, time-weighted over the expert GEMMs -- since nvidia-smi's 50 ms samples
    # of a 13 ms step miss the cap; without it, nvidia-smi's median.
    gemm_clk = [(sm_in[n], prof[n][0]) for n in GEMMS if n in sm_in and n in prof and prof[n][0] > 0]
    gemm_mhz = sum(m * t for m, t in gemm_clk) / sum(t for _, t in gemm_clk) if gemm_clk else None
    clk["gemm_sm_mhz"] = gemm_mhz
    clk["sm_mhz_in_kernels"] = {n: round(v, 1) for n, v in sm_in.items()}
    ref_mhz = gemm_mhz if gemm_mhz else clk.get("sm_mhz")
    at_max = bool(ref_mhz and clk.get("sm_max_mhz") and ref_mhz >= 0.97 * clk["sm_max_mhz"])
    tensor_peak = pk["tensor_burst"] if at_max else pk["tensor"]
    # the analytical resource model's roofline prediction for this step; the model's tensor rate is
    # the burst figure whatever the regime (its GEMM efficiency was calibrated against it)
    from mixture_experts_layer_10_gb300 import resource_model
    pred = resource_model.predict_ms(cfg, pk["tensor_burst"], pk["hbm"], N=n_kept, kept_rows=kept_real)
    cal = resource_model.predict_ms_calibrated(cfg, pk["tensor_burst"], pk["hbm"], N=n_kept, kept_rows=kept_real,
                                               counts=[int(c) for c in counts_h])
    model_line = {"predicted_ms": pred["step_ms"], "measured_over_predicted": ms / pred["step_ms"],
                  "calibrated_ms": cal["step_ms"], "measured_over_calibrated": ms / cal["step_ms"],
                  "memory_bytes": resource_model.memory(cfg)}
    tensor_kind = ("bf16_tflops (burst, %s): the GEMMs' SM clock held at max in the timed region" if at_max else
                   "bf16_tflops_sustained (%s): the GEMMs' SM clock below max (power cap) in the timed region"
                   ) % pk["source"]
    fp8_line = None
    if args.fp8 and not extra:
        fp8_line = fp8_forward(args, mc, cfg, x, W_r, b_r, Wg, Wu, Wd, dy, buf, N, tensor_peak, tensor_kind, pk, ms)
    kernels = {}
    gemm_flops = gemm_ms = hbm_bytes = hbm_ms = 0.0
    launches = 0
    for kname, (tot, n) in prof.items():
        if n == 0:
            continue
        launches += n
        ent = {"ms_per_step": tot / steps, "launches": n}
        if kname in GEMMS:
            rows_done = N - kept_real if kname == "gemm_bwd_recompute_swiglu" else N
            work = GEMMS[kname] * rows_done * d * f * n     # FLOPs over all launches
            ent["tflops"] = work / (tot / 1000.0) / 1e12
            ent["frac_of_measured_peak"] = ent["tflops"] / tensor_peak
            gemm_flops += work
            gemm_ms += tot
        elif kname in HBM_KERNELS or kname in ROUTER_KERNELS:
            if kname == "dispatch_gather" and cfg.get("gather_in_gemm"):   # tables, row tokens, row gates
                work = steps * (3 * 12 * T * k + 12 * N)
            elif kname == "dispatch_gather":   # fwd: x once + N rows; bwd: x and dy once + 2N rows
                work = steps * ((T + N) * d * 2 + 2 * (T + N) * d * 2 + 3 * 12 * T * k)
            elif kname == "combine":
                work = n * ((N + T) * d * 2 + 8 * T * k)
            elif kname == "combine_bwd":   # expert rows + the router term row in, dx out, slot indices
                work = n * ((N + 2 * T) * d * 2 + 4 * T * k)
            elif kname == "route_fwd":   # x once and W_r in; idx, gates and (kept for the backward) logits out
                work = n * (T * d * 2 + d * E * 4 + T * k * 8 + (0 if cfg.get("renorm") else T * E * 4))
            else:   # router_dlogits: idx, gates, dgates (and the kept logits) in; dl fp32 and bf16 rows out
                Ep = (E + 63) // 64 * 64
                work = n * (T * k * 12 + (0 if cfg.get("renorm") else T * E * 4) + T * E * 4 + T * Ep * 2)
            ent["gbs"] = work / (tot / 1000.0) / 1e9
            ent["frac_of_measured_peak"] = ent["gbs"] / pk["hbm"]
            if kname in HBM_KERNELS:
                hbm_bytes += work
                hbm_ms += tot
        kernels[kname] = ent
    dom = max(kernels, key=lambda n: kernels[n]["ms_per_step"])
    dom_n = kernels[dom]["launches"]
    if dom in GEMMS:
        per_launch = GEMMS[dom] * N * d * f
        achieved = per_launch / (kernels[dom]["ms_per_step"] * steps / dom_n / 1000.0) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": tensor_peak,
                "unit": "TFLOP/s", "frac": achieved / tensor_peak, "peak_kind": tensor_kind,
                "frac_of_burst": achieved / pk["tensor_burst"], "frac_of_sustained": achieved / pk["tensor"],
                "sm_mhz_in_kernel": sm_in.get(dom), "work_per_launch": per_launch}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": kernels[dom].get("gbs"), "peak": pk["hbm"],
                "unit": "GB/s", "frac": kernels[dom].get("frac_of_measured_peak")}
    roof["traffic"] = recorded_traffic(dom, name)

    value = world * T / (ms / 1000.0)
    over = args.tokens or args.experts or args.topk
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": DESCR[name] + ("" if not over or extra else f" with T={T}, E={E}, k={k} overridden"),
                   "T": T, "d_model": d, "d_ff": f, "E": E, "k": k,
                   "n_shared": S, "global_batch": world * T, "parallelism": f"replicas x{world}",
                   "l2": "no flush: each step streams > L2 (expert weights alone %.2f GB)"
                         % (3 * G * d * f * 2 / 1e9),
                   "rows_per_step": N, "load_max_over_mean": load_max_over_mean,
                   "keep_rows": keep, "kept_rows": kept_real, "gather_in_gemm": cfg.get("gather_in_gemm", 0),
                   "kept_activation_bytes": keep * f * 2 * 2, "keep_budget_bytes": keep_budget,
                   "expert_weights": "seeded on the device" if extra else "synth (seeded, host)"},
        "cuda_graph": graph,
        "model": model_line,
        "fp8_forward": fp8_line,
        "e2e": {"value": world * T / (ms_e2e / 1000.0), "unit": "tokens/s", "ms_per_step": ms_e2e,
                "h2d_bytes_per_step": 2 * T * d * 2, "d2h_bytes_per_step": 2 * T * d * 2},
        "roofline": roof,
        "expert_gemm": {"tflops": gemm_flops / (gemm_ms / 1000.0) / 1e12 if gemm_ms else None,
                        "frac_of_measured_peak": (gemm_flops / (gemm_ms / 1000.0) / 1e12 / tensor_peak)
                        if gemm_ms else None},
        "dispatch_combine": {"gbs": hbm_bytes / (hbm_ms / 1000.0) / 1e9 if hbm_ms else None,
                             "frac_of_measured_peak": (hbm_bytes / (hbm_ms / 1000.0) / 1e9 / pk["hbm"])
                             if hbm_ms else None},
        "kernels": kernels,
        "gpu_launches": launches,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not extra:
        n, dt = oracle_sample(inp, cfg, args.cpu_tokens)
        line["cpu_baseline"] = {"value": n / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"{n} seeded tokens of the same workload, fp64 fwd + bwd "
                                          f"(weight-gradient products included), {dt:.1f} s"}
    del buf, x, dy, Wg, Wu, Wd, dWg, dWu, dWd, xin, dyin, yout, dxout
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


def compact(line):
    """The per-workload record carried on the headline line."""
    k = line["kernels"]
    router = {n: {"us": 1000 * k[n]["ms_per_step"], "frac_of_hbm": k[n].get("frac_of_measured_peak")}
              for n in ROUTER_KERNELS if n in k}
    return {"workload": line["config"]["workload"], "value": line["value"], "unit": line["unit"],
            "ms_per_step": line["ms_per_step"], "steps": line["steps"], "warmup": line["warmup"],
            "e2e": {"value": line["e2e"]["value"], "ms_per_step": line["e2e"]["ms_per_step"]},
            "cuda_graph_ms": line["cuda_graph"].get("ms_per_step"),
            "roofline": {kk: line["roofline"].get(kk) for kk in ("kernel", "bound", "achieved", "peak", "unit", "frac",
                                                                 "frac_of_burst", "sm_mhz_in_kernel")},
            "expert_gemm_frac": line["expert_gemm"]["frac_of_measured_peak"],
            "dispatch_combine_frac": line["dispatch_combine"]["frac_of_measured_peak"],
            "gather_frac": k.get("dispatch_gather", {}).get("frac_of_measured_peak"),
            "combine_frac": k.get("combine", {}).get("frac_of_measured_peak"),
            "router": router,
            "model_measured_over_predicted": line["model"]["measured_over_predicted"],
            "model_measured_over_calibrated": line["model"]["measured_over_calibrated"],
            "load_max_over_mean": line["config"]["load_max_over_mean"],
            "gpu_launches": line["gpu_launches"],
            "clocks": {kk: line["clocks"].get(kk) for kk in ("sm_mhz", "sm_max_mhz", "reasons", "samples",
                                                             "gemm_sm_mhz")}}


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return

    import torch
    import torch.distributed as dist

    import mixture_experts_layer_10_gb300 as moe

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()

    moe.load()
    cfg = dict(synth.CONFIGS[args.workload])
    if args.tokens:
        cfg["T"] = args.tokens
    if args.experts:
        cfg["E"] = args.experts
    if args.topk:
        cfg["k"] = args.topk
    if args.gather_in_gemm:
        cfg["gather_in_gemm"] = 1
    line = run_workload(args, args.workload, cfg, args.steps, args.warmup, rank, world, local, barrier)
    # every other workload of the pages' families, a few steps each, as a compact record
    if not args.no_workloads and args.workload == "mixtral" and not (args.tokens or args.experts or args.topk):
        line["workloads"] = {}
        for name in synth.CONFIGS:
            if name == args.workload:
                continue
            rec = run_workload(args, name, dict(synth.CONFIGS[name]), args.workload_steps, 3, rank, world, local,
                               barrier, extra=True)
            line["workloads"][name] = compact(rec)
        # the dispatch gather fused into the expert GEMMs' operand loads, beside the default path
        for name in ("mixtral", "deepseek", "qwen3"):
            rec = run_workload(args, name, dict(synth.CONFIGS[name], gather_in_gemm=1), args.workload_steps, 3, rank,
                               world, local, barrier, extra=True)
            line["workloads"][name + "+gather_in_gemm"] = compact(rec)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
