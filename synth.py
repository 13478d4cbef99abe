"""Seeded synthetic inputs for the single-GPU MoE FFN layer.

This module is the only code shared by the fp64 oracle (``oracle/``) and the CUDA
path (``mixture_experts_layer_10_gb300``).  It holds none of the layer's arithmetic:
it draws random numbers, rounds them to their storage types (bf16 as raw ``uint16``
bits, fp32), and builds the per-expert router bias that stands in for a skewed
workload.  Nothing here routes, dispatches, multiplies or reduces.

Every tensor is drawn from its own Philox stream keyed by ``(seed, tensor id,
chunk)``, so changing one tensor's shape never shifts another tensor's values, and
large weight tensors are drawn per expert on a thread pool.

Workloads (the pages name Mixtral-, DeepSeek-, Qwen3- and GPT-OSS-shaped MoE layers
at 4K-32K sequence length; weights and data are synthetic, seed 0):

====== ===== ===== ==== == ===== == ====== ==== =====================
name   T     d     E    k  f     S  renorm cf   routing
====== ===== ===== ==== == ===== == ====== ==== =====================
tiny   256   128   8    2  256   0  0      0    unbiased
mixtral 8192 4096  8    2  14336 0  0      0    unbiased
deepseek 16384 2048 64  6  1408  2  1      0    unbiased, 2 shared
qwen3  32768 2048  128  8  768   0  0      0    Zipf(1.2) bias
gptoss 65536 2880  128  4  2880  0  0      1.25 unbiased, capacity
====== ===== ===== ==== == ===== == ====== ==== =====================

Distributions: x ~ N(0,1) -> bf16; W_r ~ N(0, 1/d) fp32; W_gate, W_up ~ N(0, 1/d)
-> bf16; W_down ~ N(0, 1/f) -> bf16; dy ~ N(0,1) -> bf16.  All roundings to bf16 are
round-to-nearest-even.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CONFIGS = {
    "tiny": dict(T=256, d=128, E=8, k=2, f=256, S=0, renorm=0, cf=0.0, zipf=False),
    "mixtral": dict(T=8192, d=4096, E=8, k=2, f=14336, S=0, renorm=0, cf=0.0, zipf=False),
    "deepseek": dict(T=16384, d=2048, E=64, k=6, f=1408, S=2, renorm=1, cf=0.0, zipf=False),
    "qwen3": dict(T=32768, d=2048, E=128, k=8, f=768, S=0, renorm=0, cf=0.0, zipf=True),
    "gptoss": dict(T=65536, d=2880, E=128, k=4, f=2880, S=0, renorm=0, cf=1.25, zipf=False),
}

# One stream id per tensor so that shapes never shift one another's values.
_TID = {"x": 1, "W_r": 2, "W_gate": 3, "W_up": 4, "W_down": 5, "dy": 6,
        "zipf_order": 7, "aux": 8}

ZIPF_S = 1.2


def make_config(name: str, **over) -> dict:
    """A copy of a named workload with fields overridden (for small parity cases)."""
    cfg = dict(CONFIGS[name])
    cfg.update(over)
    return cfg


def _rng(seed: int, tid: int, chunk: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, tid, chunk])))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return the raw bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bits to float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_f32(seed: int, name_or_tid, shape, std: float, chunk: int = 0) -> np.ndarray:
    tid = _TID[name_or_tid] if isinstance(name_or_tid, str) else int(name_or_tid)
    n = int(np.prod(shape))
    z = _rng(seed, tid, chunk).standard_normal(n, dtype=np.float32)
    z *= np.float32(std)
    return z.reshape(shape)


def normal_bf16(seed: int, name_or_tid, shape, std: float, chunk: int = 0) -> np.ndarray:
    return f32_to_bf16_bits(normal_f32(seed, name_or_tid, shape, std, chunk))


def _per_expert_bf16(seed: int, name: str, G: int, rows: int, cols: int, std: float,
                     threads: int) -> np.ndarray:
    out = np.empty((G, rows, cols), dtype=np.uint16)

    def one(g):
        out[g] = normal_bf16(seed, name, (rows, cols), std, chunk=g)

    if threads > 1 and G > 1:
        with ThreadPoolExecutor(max_workers=min(threads, G)) as ex:
            list(ex.map(one, range(G)))
    else:
        for g in range(G):
            one(g)
    return out


def zipf_bias(seed: int, E: int, s: float = ZIPF_S) -> np.ndarray:
    """Per-expert router bias 2*ln(p_r) for Zipf(s) popularity p_r over a seeded order.

    p_r is proportional to r**(-s) for ranks r = 1..E (normalised); the expert that gets
    rank r is pi(r) for a seeded random permutation pi.
    """
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** (-s)
    p /= p.sum()
    order = _rng(seed, _TID["zipf_order"], 0).permutation(E)
    b = np.empty(E, dtype=np.float64)
    b[order] = 2.0 * np.log(p)
    return b.astype(np.float32)


def capacity(cfg: dict) -> int:
    """Per-expert capacity ceil(cf*T*k/E); a large sentinel when dropless (cf <= 0)."""
    if cfg["cf"] <= 0:
        return 1 << 30
    return int(math.ceil(cfg["cf"] * cfg["T"] * cfg["k"] / cfg["E"]))


def make_inputs(cfg: dict, seed: int = 0, parts=("x", "router", "experts", "dy"),
                threads: int | None = None) -> dict:
    """Draw the layer's inputs for one workload.

    Returns a dict with (as requested by ``parts``):
      x [T,d] bf16 bits, W_r [d,E] fp32, b_r [E] fp32 or None,
      W_gate, W_up [E+S, f, d] bf16 bits, W_down [E+S, d, f] bf16 bits, dy [T,d] bf16 bits.
    """
    T, d, E, f, S = cfg["T"], cfg["d"], cfg["E"], cfg["f"], cfg["S"]
    G = E + S
    threads = threads or min(16, os.cpu_count() or 1)
    out = {}
    if "x" in parts:
        out["x"] = normal_bf16(seed, "x", (T, d), 1.0)
    if "router" in parts:
        out["W_r"] = normal_f32(seed, "W_r", (d, E), 1.0 / math.sqrt(d))
        out["b_r"] = zipf_bias(seed, E) if cfg.get("zipf") else None
    if "experts" in parts:
        out["W_gate"] = _per_expert_bf16(seed, "W_gate", G, f, d, 1.0 / math.sqrt(d), threads)
        out["W_up"] = _per_expert_bf16(seed, "W_up", G, f, d, 1.0 / math.sqrt(d), threads)
        out["W_down"] = _per_expert_bf16(seed, "W_down", G, d, f, 1.0 / math.sqrt(f), threads)
    if "dy" in parts:
        out["dy"] = normal_bf16(seed, "dy", (T, d), 1.0)
    return out


def random_assignments(seed: int, T: int, E: int, k: int, skew: float = 0.0) -> np.ndarray:
    """Distinct expert ids per token, [T,k] int32, optionally Zipf-skewed (for dispatch cases).

    Draws k distinct experts per token by sorting seeded keys; with ``skew`` > 0 the keys
    are shifted by 2*ln(Zipf popularity) so a few experts get most tokens.
    """
    rng = _rng(seed, _TID["aux"], 1)
    keys = rng.gumbel(size=(T, E))
    if skew > 0:
        keys = keys + zipf_bias(seed, E, skew).astype(np.float64)[None, :]
    idx = np.argsort(-keys, axis=1, kind="stable")[:, :k]
    return np.ascontiguousarray(idx.astype(np.int32))


def uniform_f32(seed: int, shape, lo: float, hi: float, chunk: int = 0) -> np.ndarray:
    z = _rng(seed, _TID["aux"], 100 + chunk).random(int(np.prod(shape)), dtype=np.float32)
    return (np.float32(lo) + z * np.float32(hi - lo)).reshape(shape)
