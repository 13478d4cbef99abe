"""FP8 (e4m3) expert inputs on the GPU against the oracle's quantisation step (GPU).

* the row quantiser: codes and scales bit-exact (both sides decide in fp32);
* the e4m3 gate/up projection with SwiGLU: h of every kept row against the fp64 product of the
  oracle's own codes and scales, under the bf16 output rule.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
from cases import case
from harness import check_close, from_dev, from_dev_bf16, segment_rows, to_dev, to_dev_bf16
import synth

pytestmark = pytest.mark.gpu


def _quantize_dev(moe, t):
    rows = t.numel() // t.shape[-1]
    codes = torch.empty(t.shape, dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, dtype=torch.float32, device="cuda")
    moe.moe_quantize_rows_e4m3(t, codes, scales)
    return codes, scales


@pytest.mark.parametrize("cols", [64, 192, 2880])
def test_quantize_rows_bit_exact(moe, cols):
    rng = np.random.default_rng(cols)
    v = rng.normal(0, 1, (97, cols)) * np.exp(rng.uniform(-12, 12, (97, 1)))
    v[3] = 0.0                                     # an all-zero row
    v[5, ::7] *= 1e-6                              # subnormal codes inside a row
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
