"""The FP8 (e4m3) forward on the GPU against the oracle's quantised forward (GPU).

* the row quantiser: codes and scales bit-exact (both sides decide in fp32);
* the e4m3 gate/up projection with SwiGLU and the e4m3 down projection: every kept row against the
  fp64 product of the oracle's own codes and scales, under the bf16 output rule;
* moe_layer_fwd_fp8: y on the small workloads, on constructed layers where every quantisation step
  is exact, and on sampled tokens and output channels at the Mixtral- and Qwen3-like full sizes.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
from cases import case
from harness import (check_close, check_routing, decided_tokens, from_dev, from_dev_bf16, segment_rows, to_dev,
                     to_dev_bf16)
import synth

pytestmark = pytest.mark.gpu


def _quantize_dev(moe, t):
    rows = t.numel() // t.shape[-1]
    codes = torch.empty(t.shape, dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, dtype=torch.float32, device="cuda")
    moe.moe_quantize_rows_e4m3(t, codes, scales)
    return codes, scales


@pytest.mark.parametrize("cols", [64, 192, 1024, 2880, 14336, 16384])   # 32 to 256 threads a row
def test_quantize_rows_bit_exact(moe, cols):
    rng = np.random.default_rng(cols)
    v = rng.normal(0, 1, (97, cols)) * np.exp(rng.uniform(-12, 12, (97, 1)))
    v[3] = 0.0                                     # an all-zero row
    v[5, ::7] *= 1e-6                              # subnormal codes inside a row
    v[6, ::3] = -0.0                               # signed zeros
    # quotients exactly on e4m3 rounding ties (scale 2^-5: row maximum 448 * 2^-5): ties to even
    ties = np.array([1.0625, 1.1875, -1.0625, 2.0 ** -10, 3 * 2.0 ** -10, -5 * 2.0 ** -10, 17.0, 19.0, 400.0])
    v[7] = np.resize(ties, cols) * 2.0 ** -5
    v[7, 0] = 448.0 * 2.0 ** -5
    v[8] *= 1e-30 / np.abs(v[8]).max()             # scale below 2^-80: the IEEE-division rows
    v[9] *= 1e30 / np.abs(v[9]).max()              # scale above 2^80
    bits = synth.f32_to_bf16_bits(v.astype(np.float32))
    codes, scales = _quantize_dev(moe, to_dev_bf16(bits))
    torch.cuda.synchronize()
    ref_q, ref_s = fp8.quantize_rows_e4m3(oracle.bf16_to_f64(bits).astype(np.float32))
    assert np.array_equal(from_dev(scales), ref_s)
    assert np.array_equal(from_dev(codes), ref_q)


@pytest.mark.parametrize("name", ["ragged_mixtral", "deepseek_small", "gptoss_small", "qwen_small"])
def test_gate_up_fp8(moe, name):
    c, inp, L = case(name)
    mc = moe.config_from(c)
    buf = moe.Buffers.allocate(mc)
    T, E, S, d, f, k = c["T"], c["E"], c["S"], c["d"], c["f"], c["k"]
    D = L.dispatch()
    x_perm = torch.zeros(buf.rows, d, dtype=torch.bfloat16, device="cuda")
    scratch = [torch.empty(n, dtype=torch.int32, device="cuda") for n in (E, E + 1, T * k, T * k)]
    moe.moe_dispatch(mc, to_dev(L.routing().idx.astype(np.int32)), to_dev_bf16(inp["x"]), *scratch, x_perm, buf.ws)
    x8, xs = _quantize_dev(moe, x_perm)
    g8, gs = _quantize_dev(moe, to_dev_bf16(inp["W_gate"]))
    u8, us = _quantize_dev(moe, to_dev_bf16(inp["W_up"]))
    h = torch.full((buf.rows, f), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_gate_up_fp8(mc, x8, xs, g8, gs.view(E + S, f), u8, us.view(E + S, f), h, buf.ws)
    assert moe.moe_check_error(buf.ws) == 0
    # the oracle's own quantisation of x and of every weight row
    xq, xsc = fp8.quantize_rows_e4m3(L.x.astype(np.float32))
    kept, P = segment_rows(D, T, S)
    got_h = from_dev_bf16(h)
    refs, gots = [], []
    for g in range(E + S):
        if kept[g] == 0:
            continue
        toks = D.token_of_row[D.offsets[g]:D.offsets[g + 1]] if g < E else np.arange(T)
        wg, wu, _ = L.W(g)
        gq, gsc = fp8.quantize_rows_e4m3(wg.astype(np.float32))
        uq, usc = fp8.quantize_rows_e4m3(wu.astype(np.float32))
        refs.append(fp8.gate_up_fp8(xq[toks], xsc[toks], gq, gsc, uq, usc))
        gots.append(got_h[P[g]:P[g] + kept[g]])
        assert np.all(got_h[P[g] + kept[g]:P[g + 1]] == 0), f"pad rows of segment {g}"
    check_close("h (fp8 gate/up)", np.concatenate(gots), np.concatenate(refs))


@pytest.mark.parametrize("name", ["ragged_mixtral", "deepseek_small", "gptoss_small"])
def test_down_fp8(moe, name):
    c, inp, L = case(name)
    mc = moe.config_from(c)
    buf = moe.Buffers.allocate(mc)
    T, E, S, d, f, k = c["T"], c["E"], c["S"], c["d"], c["f"], c["k"]
    D = L.dispatch()
    scratch = [torch.empty(n, dtype=torch.int32, device="cuda") for n in (E, E + 1, T * k, T * k)]
    x_perm = torch.zeros(buf.rows, d, dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch(mc, to_dev(L.routing().idx.astype(np.int32)), to_dev_bf16(inp["x"]), *scratch, x_perm, buf.ws)
    # an h of the scale SwiGLU gives, with rows of very different magnitude
    h_bits = synth.f32_to_bf16_bits(synth.normal_f32(11, 21, (buf.rows, f), 0.05)
                                    * np.exp2(np.arange(buf.rows) % 9 - 4)[:, None].astype(np.float32))
    h8, hs = _quantize_dev(moe, to_dev_bf16(h_bits))
    d8, ds = _quantize_dev(moe, to_dev_bf16(inp["W_down"]))
    o = torch.full((buf.rows, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_down_fp8(mc, h8, hs, d8, ds.view(E + S, d), o, buf.ws)
    assert moe.moe_check_error(buf.ws) == 0
    hq, hsc = fp8.quantize_rows_e4m3(oracle.bf16_to_f64(h_bits).astype(np.float32))
    kept, P = segment_rows(D, T, S)
    got_o = from_dev_bf16(o)
    refs, gots = [], []
    for g in range(E + S):
        rows = np.arange(P[g], P[g] + kept[g])
        if rows.size == 0:
            continue
        dq, dsc = fp8.quantize_rows_e4m3(L.W(g)[2].astype(np.float32))
        refs.append(fp8.down_fp8(hq[rows], hsc[rows], dq, dsc))
        gots.append(got_o[rows])
    ref = np.concatenate(refs)
    check_close("o (fp8 down)", np.concatenate(gots), ref)


def _run_fwd_fp8(moe, c, inp):
    mc = moe.config_from(c)
    buf = moe.Buffers.allocate(mc)
    T, E, S, d, f, k = c["T"], c["E"], c["S"], c["d"], c["f"], c["k"]
    q = {}
    for key in ("W_gate", "W_up", "W_down"):
        codes, scales = _quantize_dev(moe, to_dev_bf16(inp[key]))
        q[key] = (codes, scales.view(E + S, -1))
    y = torch.full((T, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    b_r = to_dev(inp["b_r"]) if inp["b_r"] is not None else None
    moe.moe_layer_fwd_fp8(mc, to_dev_bf16(inp["x"]), to_dev(inp["W_r"]), b_r, *q["W_gate"], *q["W_up"],
                          *q["W_down"], y, buf.saved, buf.ws)
    status = moe.moe_check_error(buf.ws)
    assert status == 0, moe.moe_status_string(status)
    idx = buf.saved.view(torch.int32)[:T * k].view(T, k)
    gates = buf.saved.view(torch.float32)[T * k:2 * T * k].view(T, k)
    return from_dev_bf16(y), from_dev(idx), from_dev(gates)


@pytest.mark.parametrize("name", ["tiny", "ragged_mixtral", "deepseek_small", "gptoss_small", "qwen_small",
                                  "single_expert", "k_equals_E", "max_experts", "max_shared", "router_e96_k8",
                                  "router_simt_e160", "max_d_model", "max_d_ff"])
def test_layer_fwd_fp8(moe, name):
    c, inp, L = case(name)
    _check_fwd_fp8(moe, c, inp, L)


# widths that are multiples of 64 but not of 128 (the e4m3 K blocks are 128 codes: the last one is
# half zero-filled), a single token, and a capacity of one row per expert
@pytest.mark.parametrize("over", [dict(T=160, d=2880, f=192, E=4, k=2), dict(T=150, d=192, f=2880, E=4, k=2),
                                  dict(T=1, d=64, f=64, E=4, k=2, S=1),
                                  dict(T=200, d=128, f=128, E=8, k=2, cf=1.0 / 50)])
def test_layer_fwd_fp8_shapes(moe, over):
    c = dict(T=0, d=0, f=0, E=0, k=0, S=0, renorm=0, cf=0.0, zipf=False)
    c.update(over)
    inp = synth.make_inputs(c, seed=4)
    _check_fwd_fp8(moe, c, inp, oracle.Layer(inp, c))


def _check_fwd_fp8(moe, c, inp, L):
    y, idx, gates = _run_fwd_fp8(moe, c, inp)
    same = check_routing(idx, gates, L.routing(), c["k"])
    if not same.all():
        assert c["cf"] <= 0, "capacity workloads must route identically"
    rows = np.flatnonzero(same)
    y_ref = fp8.layer_forward_fp8(L)
    check_close("y (fp8 forward)", y[rows], y_ref[rows], float(np.abs(y_ref).max()))


@pytest.mark.parametrize("variant", [dict(), dict(S=0, renorm=True, k=3), dict(cf=0.6, S=2)])
def test_layer_fwd_fp8_lossless(moe, variant):
    # every quantisation step exact: the GPU forward equals the exact layer up to its own fp32
    # sums and the bf16 output
    from test_oracle_fp8 import _lossless_layer
    L = _lossless_layer(**variant)
    c = dict(L.cfg)
    y, idx, gates = _run_fwd_fp8(moe, c, L.inp)
    assert check_routing(idx, gates, L.routing(), c["k"]).all()
    y_ref, _ = L.forward()
    check_close("y (lossless fp8 forward)", y, y_ref)


@pytest.mark.slow
@pytest.mark.parametrize("name,n_tok", [("mixtral", 16), ("qwen3", 4), ("deepseek", 4), ("gptoss", 4)])
def test_layer_fwd_fp8_full_size(moe, name, n_tok):
    """The FP8 forward at the workload's full size, as bench.py --fp8 runs it: y of sampled tokens
    and output channels against the oracle, one token at a time.  The oracle quantises only the
    experts the sample visits, so the Mixtral-like sample is drawn from the tokens routed to the
    most common expert pair.  With a capacity, a slot's survival depends on every earlier token's
    routing, so the sample comes from the tokens before the first routing difference."""
    cfg = synth.CONFIGS[name]
    inp = synth.make_inputs(cfg, seed=0)
    L = oracle.Layer(inp, cfg)
    y, idx, gates = _run_fwd_fp8(moe, cfg, inp)
    R = L.routing()
    same = check_routing(idx, gates, R, cfg["k"])
    order_ok, _ = decided_tokens(R.logits, cfg["k"])
    agree = same & order_ok
    if cfg["cf"] > 0 and not same.all():
        agree[int(np.flatnonzero(~same)[0]):] = False
    pool = np.flatnonzero(agree)
    if name == "mixtral":
        pairs = np.sort(R.idx[pool], axis=1)
        key = pairs[:, 0] * cfg["E"] + pairs[:, 1]
        pool = pool[key == np.bincount(key).argmax()]
    rng = np.random.default_rng(9)
    toks = np.sort(rng.choice(pool, size=n_tok, replace=False))
    cols = np.sort(rng.choice(cfg["d"], size=64, replace=False))
    ref = fp8.token_outputs_fp8(L, toks, cols)
    check_close("y (fp8 forward, full size)", y[toks][:, cols], ref)
