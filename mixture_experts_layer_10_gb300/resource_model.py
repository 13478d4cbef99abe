"""Analytical resource model of one MoE layer step (forward + backward) on one GPU.

Piper's explainer (planner section) predicts each stage's memory and compute from the model shape
and checks the prediction against measurement; this is the same idea for the single-GPU layer
built here.  From the configuration alone (and, optionally, the number of routed rows the experts
really see) it gives:

* memory: the workspace and `saved` bytes the library asks for, the caller's tensors, and the
  activation bytes kept between forward and backward;
* work per kernel: FLOPs for the tensor-core kernels, algorithmic HBM bytes for the gather/combine
  kernels (the same definitions bench.py reports against);
* a roofline time per kernel, max(FLOPs / tensor rate, bytes / HBM rate) plus a fixed launch cost,
  summed into a predicted step time that bench.py sets beside the measured one.

Host arithmetic only: nothing here runs on the GPU or calls the library.
"""
from __future__ import annotations

import math

ROW_TILE = 256          # expert segments are padded to this many rows (include/moe.h)
LAUNCH_US = 4.0         # fixed cost per kernel launch on the stream, microseconds


def padded_rows(T: int, k: int, E: int, S: int) -> int:
    """Row capacity of the expert-ordered buffers: every routed segment rounded up to the tile, in
    the worst case E - 1 extra tiles' worth of padding, plus S shared segments of T rows."""
    routed = math.ceil((T * k + (ROW_TILE - 1) * E) / ROW_TILE) * ROW_TILE
    return routed + S * math.ceil(T / ROW_TILE) * ROW_TILE


def router_n(E: int, k: int) -> int:
    """Columns the router's logit product computes per token: E <= 32 (k <= 8) stacks the three bf16
    parts of W_r along N (E rounded to 8/16/32, times three, rounded to 16); up to 128 experts
    the parts take E rounded to 64 each; beyond, the fp32 product computes E."""
    if E <= 32 and k <= 8:
        eb = 8 if E <= 8 else 16 if E <= 16 else 32
        return math.ceil(3 * eb / 16) * 16
    if E <= 128 and k <= 8:
        return 3 * math.ceil(E / 64) * 64
    return E


def kept_rows(cfg: dict) -> int:
    """keep_rows as the library applies it: rounded down to the pair tile, at most all rows."""
    T, E, k, S = cfg["T"], cfg["E"], cfg["k"], cfg.get("S", 0)
    return min(cfg.get("keep_rows", 0) // ROW_TILE * ROW_TILE, padded_rows(T, k, E, S))


def keep_rows_for_budget(cfg: dict, budget_bytes: int) -> int:
    """The largest keep_rows whose kept a and b (4 d_ff bytes a row) fit in the budget."""
    T, f, E, k, S = cfg["T"], cfg["f"], cfg["E"], cfg["k"], cfg.get("S", 0)
    return min(budget_bytes // (4 * f) // ROW_TILE * ROW_TILE, padded_rows(T, k, E, S))


def memory(cfg: dict) -> dict:
    """Bytes of device memory one layer instance needs, by owner."""
    T, d, f, E, k, S = cfg["T"], cfg["d"], cfg["f"], cfg["E"], cfg["k"], cfg.get("S", 0)
    G = E + S
    Ep = math.ceil(E / 64) * 64
    rows = padded_rows(T, k, E, S)
    ndg = 2 * math.ceil(f / 128)
    per_row = (2 * d + 4 * f + d) * 2 + (4 + 4 + 4 * ndg)   # x/dY/O planes, four d_ff planes, metadata
    workspace = (rows * per_row + T * k * 12 + T * E * 4 + T * Ep * 2 + 4 * d * Ep * 2
                 + math.ceil(T * k / 4096) * E * 4)
    keep = kept_rows(cfg)
    saved = 8 * T * k                  # idx, gates
    if not cfg.get("renorm", 0):       # the logits, for the backward's softmax
        saved = math.ceil(saved / 256) * 256 + T * E * 4
    if keep:
        saved = math.ceil(saved / 256) * 256 + keep * f * 2 * 2
    return {
        "padded_rows": rows,
        "workspace": workspace,
        "saved": saved,                   # idx, gates, logits and the kept a, b: what lives fwd -> bwd
        "weights": 3 * G * d * f * 2 + d * E * 4,
        "weight_grads": 3 * G * d * f * 2 + d * E * 4,
        "token_tensors": 4 * T * d * 2,   # x, y, dy, dx
        "kept_activations": keep * f * 2 * 2,
    }


def work(cfg: dict, N: int | None = None, kept_rows: int = 0) -> dict:
    """FLOPs and algorithmic HBM bytes per kernel of one forward + backward step.

    N is the number of routed rows the experts see (kept assignments); by default T*k (dropless).
    kept_rows are rows whose a, b the forward keeps, which the recompute GEMM then skips."""
    T, d, f, E, k, S = cfg["T"], cfg["d"], cfg["f"], cfg["E"], cfg["k"], cfg.get("S", 0)
    N = T * k if N is None else N
    R = N + S * T                                      # rows the experts see
    Ep = math.ceil(E / 64) * 64
    nr = router_n(E, k)
    logits = 0 if cfg.get("renorm", 0) else T * E * 4   # kept by the forward for the backward
    out = {
        "route_fwd": {"flops": 2 * T * d * nr, "bytes": T * d * 2 + logits},
        "dispatch_gather": {"flops": 0, "bytes": 3 * (T + R) * d * 2 + 36 * T * k},
        "gemm_gate_up_swiglu": {"flops": 4 * R * d * f, "bytes": 0},
        "gemm_down": {"flops": 2 * R * d * f, "bytes": 0},
        "combine": {"flops": 0, "bytes": (R + T) * d * 2 + 8 * T * k},
        "gemm_bwd_dgrad_down": {"flops": 2 * R * d * f, "bytes": 0},
        "gemm_bwd_recompute_swiglu": {"flops": 4 * (R - kept_rows) * d * f, "bytes": 0},
        "gemm_wgrad": {"flops": 6 * R * d * f, "bytes": 0},
        "gemm_dgrad_x": {"flops": 4 * R * d * f, "bytes": 0},
        "router_dlogits": {"flops": 0, "bytes": 12 * T * k + logits + T * E * 4 + T * Ep * 2},
        "router_dwr": {"flops": 2 * T * d * Ep, "bytes": T * d * 2},
        "gemm_router_dx": {"flops": 2 * T * d * Ep, "bytes": T * d * 2},
        "combine_bwd": {"flops": 0, "bytes": (R + 2 * T) * d * 2 + 4 * T * k},
    }
    if kept_rows:
        out["swiglu_bwd_kept"] = {"flops": 0, "bytes": 6 * kept_rows * f * 2}
    return out


def gemm_flops(cfg: dict, N: int | None = None, kept_rows: int = 0) -> int:
    """Expert GEMM FLOPs of one step: 22 (N + S T) d f with full recompute."""
    return sum(v["flops"] for n, v in work(cfg, N, kept_rows).items() if n.startswith("gemm_")
               and n != "gemm_router_dx")


def predict_ms(cfg: dict, tensor_tflops: float, hbm_gbs: float, N: int | None = None,
               kept_rows: int = 0, launches: int = 17) -> dict:
    """Roofline time per kernel and the step total, in milliseconds."""
    per = {}
    for name, w in work(cfg, N, kept_rows).items():
        t_tc = w["flops"] / (tensor_tflops * 1e12)
        t_hbm = w["bytes"] / (hbm_gbs * 1e9)
        per[name] = 1e3 * max(t_tc, t_hbm)
    total = sum(per.values()) + launches * LAUNCH_US / 1e3
    return {"step_ms": total, "per_kernel_ms": per}


# Calibration of the step-time model on GB300 (one GPU, kernels timed inside the bench's step).  The
# roofline above leaves out what the kernels cannot avoid or have not removed: the expert GEMMs run
# over padded rows at a fraction of the peak, the HBM kernels at a fraction of the copy bandwidth,
# the dispatch scan is latency (a decoupled look-back), and the routers have fixed costs.  The GEMM
# and HBM fractions are the Mixtral-like step's live figures; the router and scan constants come
# from the routers' and the scan's own timings at several shapes.  Other workloads are predictions.
# The GEMM fraction counts the pad rows' MMAs: 0.95 over padded rows is ~0.90 over routed rows.
EFF_GEMM = 0.95          # expert pair GEMMs, of the tensor peak passed in, over padded rows
EFF_HBM = 0.85           # gather / combine kernels, of the copy bandwidth passed in
SCAN_US = 30.0           # one dispatch scan (two per step)
ROUTER_FIXED_US = 12.0   # streaming router (E <= 32): setup, first loads, cross-CTA finish, per pass
ROUTER_TILE_US = 16.0    # per-tile router (32 < E <= 128): softmax / top-k epilogue of a 128-token tile
SMALL_US = 10.0          # the small reductions (gate partials, router partials) per launch
NUM_SMS = 152


def padded_routed_rows(counts, row_tile: int = ROW_TILE) -> int:
    """Rows the expert GEMMs run over for per-expert row counts: each expert's rows rounded up to the
    tile (an expert with none takes no rows)."""
    return int(sum(math.ceil(int(c) / row_tile) * row_tile for c in counts))


def predict_ms_calibrated(cfg: dict, tensor_tflops: float, hbm_gbs: float, N: int | None = None,
                          kept_rows: int = 0, counts=None) -> dict:
    """Step time from the calibrated model: per kernel, its work at the efficiency the kernel class
    reaches on GB300, plus its fixed costs.  counts: the routed rows of each expert (the padded
    rows then follow them); without them every expert gets an equal share."""
    T, d, f, E, k, S = cfg["T"], cfg["d"], cfg["f"], cfg["E"], cfg["k"], cfg.get("S", 0)
    N = T * k if N is None else N
    if counts is None:
        counts = [N // E + (1 if e < N % E else 0) for e in range(E)]
    R = N + S * T
    Rpad = padded_routed_rows(counts) + S * math.ceil(T / ROW_TILE) * ROW_TILE
    w = work(cfg, N, kept_rows)
    tc, bw = tensor_tflops * 1e12, hbm_gbs * 1e9
    per = {}
    for name, v in w.items():
        if name.startswith("gemm_") and name != "gemm_router_dx":
            per[name] = 1e3 * v["flops"] * (Rpad / max(R, 1)) / (EFF_GEMM * tc)
        elif name in ("dispatch_gather", "combine", "combine_bwd", "swiglu_bwd_kept"):
            per[name] = 1e3 * v["bytes"] / (EFF_HBM * bw)
    Ep = math.ceil(E / 64) * 64
    per["router_dlogits"] = 1e3 * (w["router_dlogits"]["bytes"] / (EFF_HBM * bw) + SMALL_US * 1e-6)
    for name in ("route_fwd",):
        if E <= 32 and k <= 8:
            t = T * d * 2 / (EFF_HBM * bw) + ROUTER_FIXED_US * 1e-6
        elif E <= 128 and k <= 8:
            tiles = math.ceil(T / 128)
            waves = math.ceil(tiles / NUM_SMS)
            mma = 2 * 128 * 3 * Ep * d / (tc / NUM_SMS)
            t = waves * (mma + ROUTER_TILE_US * 1e-6)
        else:   # the SIMT fp32 kernels
            t = 2 * T * d * E / (tc / 16) + T * d * 2 / bw
        per[name] = 1e3 * t
    for name in ("router_dwr", "gemm_router_dx"):   # small GEMMs over T (K or M) and Ep
        per[name] = 1e3 * max(2 * T * d * Ep / (0.5 * tc), T * d * 2 / (0.5 * bw))
    per["dispatch_scan"] = 2 * SCAN_US * 1e-3
    per["small_reductions"] = 2 * SMALL_US * 1e-3
    total = sum(per.values()) + len(per) * LAUNCH_US * 1e-3 / 2
    return {"step_ms": total, "per_kernel_ms": per, "padded_rows": Rpad}


def work_forward(cfg: dict, N: int | None = None, fp8: bool = False) -> dict:
    """FLOPs and algorithmic HBM bytes per kernel of the forward alone, in bf16 (moe_layer_fwd) or
    with e4m3 expert GEMMs (moe_layer_fwd_fp8: the token rows quantised once, their codes and row
    scales gathered, h quantised per row between the projections).  FP8 FLOPs are reported under
    "fp8_flops" so that the prediction can run them at the FP8 tensor rate."""
    T, d, f, E, k, S = cfg["T"], cfg["d"], cfg["f"], cfg["E"], cfg["k"], cfg.get("S", 0)
    N = T * k if N is None else N
    R = N + S * T
    logits = 0 if cfg.get("renorm", 0) else T * E * 4   # kept for the backward
    out = {"route_fwd": {"flops": 2 * T * d * router_n(E, k), "bytes": T * d * 2 + logits}}
    if fp8:
        out["quantize_e4m3 (x)"] = {"flops": 0, "bytes": T * d * 3 + 4 * T}
        out["dispatch_gather"] = {"flops": 0, "bytes": (T + R) * d + 8 * R + 12 * T * k}
        out["gemm_gate_up_fp8"] = {"flops": 0, "fp8_flops": 4 * R * d * f, "bytes": 0}
        out["quantize_e4m3 (h)"] = {"flops": 0, "bytes": R * f * 3 + 4 * R}
        out["gemm_down_fp8"] = {"flops": 0, "fp8_flops": 2 * R * d * f, "bytes": 0}
    else:
        out["dispatch_gather"] = {"flops": 0, "bytes": (T + R) * d * 2 + 12 * T * k}
        out["gemm_gate_up_swiglu"] = {"flops": 4 * R * d * f, "bytes": 0}
        out["gemm_down"] = {"flops": 2 * R * d * f, "bytes": 0}
    out["combine"] = {"flops": 0, "bytes": (R + T) * d * 2 + 8 * T * k}
    return out


def predict_forward_ms(cfg: dict, tensor_tflops: float, hbm_gbs: float, N: int | None = None,
                       fp8: bool = False) -> dict:
    """Roofline time of the forward alone; FP8 GEMMs at twice the bf16 tensor rate (the nominal
    ratio of the dense FP8 and bf16 peaks)."""
    per = {}
    work_ = work_forward(cfg, N, fp8)
    for name, w in work_.items():
        t_tc = (w["flops"] + w.get("fp8_flops", 0) / 2) / (tensor_tflops * 1e12)
        t_hbm = w["bytes"] / (hbm_gbs * 1e9)
        per[name] = 1e3 * max(t_tc, t_hbm)
    total = sum(per.values()) + (len(work_) + 1) * LAUNCH_US / 1e3   # + the dispatch scan
    return {"step_ms": total, "per_kernel_ms": per}
