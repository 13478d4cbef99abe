"""Small and medium parity workloads (seconds for the oracle, several tiles and ragged tails).

Each case is shaped like one of the pages' workload families (Mixtral-, DeepSeek-, Qwen3- and
GPT-OSS-like layers) but small: segments of 1-3 M tiles with ragged ends, d_model and d_ff that are
multiples of 64 but not of 128 or 256, shared experts with renormalised gates, a Zipf-skewed router
with empty experts, and a capacity that drops slots.
"""
from __future__ import annotations

import functools

import oracle
import synth

CASES = {
    "tiny": dict(synth.CONFIGS["tiny"]),
    "ragged_mixtral": dict(T=1000, d=320, E=8, k=2, f=384, S=0, renorm=0, cf=0.0, zipf=False),
    "deepseek_small": dict(T=512, d=256, E=16, k=4, f=192, S=2, renorm=1, cf=0.0, zipf=False),
    "qwen_small": dict(T=777, d=128, E=32, k=4, f=128, S=0, renorm=0, cf=0.0, zipf=True),
    "gptoss_small": dict(T=600, d=192, E=16, k=4, f=192, S=0, renorm=0, cf=1.25, zipf=True),
    "single_expert": dict(T=100, d=64, E=1, k=1, f=64, S=0, renorm=0, cf=0.0, zipf=False),
    "k_equals_E": dict(T=130, d=128, E=4, k=4, f=128, S=1, renorm=1, cf=0.0, zipf=False),
    # tensor-core router shapes: E not a multiple of 64 (padded logit columns), k = 8, a router
    # bias, and d_model = 320 (five 64-wide K blocks: one full 256-wide K slice and a short one)
    "router_e96_k8": dict(T=333, d=320, E=96, k=8, f=64, S=0, renorm=0, cf=0.0, zipf=True),
    # tensor-core forward with renormalised gates (the backward then needs no logits)
    "router_e64_renorm": dict(T=257, d=256, E=64, k=6, f=128, S=1, renorm=1, cf=0.0, zipf=False),
    # the fp32 SIMT router: more than 128 experts, and more than 8 experts per token
    "router_simt_e160": dict(T=300, d=128, E=160, k=4, f=64, S=0, renorm=0, cf=0.0, zipf=True),
    "router_simt_k10": dict(T=200, d=192, E=24, k=10, f=64, S=0, renorm=1, cf=0.0, zipf=False),
    # more slots per token than a warp has lanes (k = 40): the layer backward's dlogits then walks
    # each token's slots in every lane instead of holding one slot per lane
    "router_simt_k40": dict(T=70, d=128, E=64, k=40, f=64, S=0, renorm=0, cf=0.0, zipf=False),
    # limits: the most routed experts (256), and the most shared experts (8) at the narrowest widths
    "max_experts": dict(T=700, d=64, E=256, k=2, f=64, S=0, renorm=0, cf=0.0, zipf=False),
    "max_shared": dict(T=300, d=64, E=4, k=1, f=64, S=8, renorm=1, cf=0.0, zipf=False),
    # the widest rows the library accepts: d_model = 16384, and d_ff = 16384
    "max_d_model": dict(T=96, d=16384, E=4, k=2, f=128, S=1, renorm=0, cf=0.0, zipf=False),
    "max_d_ff": dict(T=96, d=128, E=4, k=2, f=16384, S=1, renorm=0, cf=0.0, zipf=False),
}

FAST = ["tiny", "ragged_mixtral", "deepseek_small", "qwen_small", "gptoss_small"]


@functools.lru_cache(maxsize=None)
def case(name: str, seed: int = 0):
    cfg = dict(CASES[name])
    inp = synth.make_inputs(cfg, seed=seed)
    return cfg, inp, oracle.Layer(inp, cfg)
