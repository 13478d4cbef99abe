"""FP8 (e4m3) quantisation step, the quantised forward and the quantised backward, for the oracle.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only tests, ``__graft_entry__.smoke()`` and bench.py's CPU legs
use it.

The pages name mixed-precision / quantised experts only as a direction ("MoEBlaze" summary,
limitations and future work); they fix no format.  The plainest reading taken here:

* the format is OCP FP8 E4M3 (the "fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3
  mantissa bits; no infinities; the largest finite magnitude is 448 (exponent 15, mantissa 6);
  exponent field 0 holds the subnormals m * 2^-9; pattern S.1111.111 is NaN and never produced;
* a row of values v (bf16 widened exactly) is scaled by s = amax / 448 with amax = max |v| over
  the row, computed in fp32 (s = 1 when the row is all zero); each element is then v / s in fp32,
  rounded to the nearest e4m3 value with ties to the even mantissa, and saturated to +-448;
* an activation row and a weight row (one output channel) are quantised this way, so
  x . w ~= s_x s_w (q_x . q_w), exactly the fp64 product of the decoded codes and the scales.
* in the forward the SwiGLU output h is held in bf16 between the two projections (the precision
  of every other intermediate of the layer) and quantised per row like x; W_down is quantised per
  row, one scale per output channel of d_model; the router stays in fp32.

Both rounding decisions (the fp32 division and the e4m3 rounding) are taken in fp32, as the
kernels take them.
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import as_f64, combine, f64_to_bf16_value, router_backward, router_backward_logits

E4M3_MAX = 448.0
_MIN_NORMAL_EXP = -6          # smallest normal: 2^-6
_MANT_BITS = 3


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """float64 values of e4m3 codes (NaN patterns decode to NaN)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = sign * np.ldexp(1.0 + m / 8.0, e - 7)
    sub = sign * np.ldexp(m / 8.0, _MIN_NORMAL_EXP)
    v = np.where(e == 0, sub, normal)
    return np.where((e == 15) & (m == 7), np.nan, v)


def e4m3_encode_rne(v: np.ndarray) -> np.ndarray:
    """Nearest e4m3 code to each float (float32 or float64 values), ties to even mantissa,
    magnitudes above 448 saturated to 448."""
    v = np.asarray(v, dtype=np.float64)
    neg = np.signbit(v)
    a = np.minimum(np.abs(v), E4M3_MAX)
    # quantum of the binade (subnormals share the smallest normal binade's quantum 2^-9)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, _MIN_NORMAL_EXP)
    q = np.ldexp(1.0, (e - _MANT_BITS).astype(np.int64))
    r = np.rint(a / q) * q                      # np.rint rounds half to even
    r = np.minimum(r, E4M3_MAX)
    # encode the rounded magnitude (it may have moved up a binade)
    with np.errstate(divide="ignore"):
        er = np.floor(np.log2(np.where(r > 0, r, 1.0)))
    is_sub = r < np.ldexp(1.0, _MIN_NORMAL_EXP)
    exp_field = np.where(is_sub, 0, er + 7).astype(np.int64)
    mant = np.where(is_sub, r / np.ldexp(1.0, _MIN_NORMAL_EXP - _MANT_BITS),
                    r / np.ldexp(1.0, (er - _MANT_BITS).astype(np.int64)) - 8.0)
    code = (exp_field << 3) | np.rint(mant).astype(np.int64)
    code = np.where(r == 0, 0, code)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


def quantize_rows_e4m3(rows: np.ndarray):
    """Per-row scaling and e4m3 codes of a [n, width] array of exact fp32 values (bf16 inputs).

    Returns (codes uint8 [n, width], scales float32 [n])."""
    v = np.asarray(rows, dtype=np.float32)
    amax = np.max(np.abs(v), axis=1) if v.shape[1] else np.zeros(v.shape[0], np.float32)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    scaled = (v / scale[:, None]).astype(np.float32)   # fp32 division, round to nearest
    return e4m3_encode_rne(scaled), scale


def dequantize_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """float64 values the quantised rows stand for: code value times the row's scale (exact)."""
    return e4m3_decode(codes) * np.asarray(scales, np.float64)[:, None]


def gate_up_fp8(xq: np.ndarray, xs: np.ndarray, gq: np.ndarray, gs: np.ndarray, uq: np.ndarray,
                us: np.ndarray) -> np.ndarray:
    """h = silu(a) * b for quantised rows: a = (s_x q_x) (s_g q_g)^T, b likewise with the up rows,
    in float64.  xq [n, d] codes, xs [n]; gq, uq [f, d] codes, gs, us [f] (one expert)."""
    x = dequantize_rows(xq, xs)
    a = x @ dequantize_rows(gq, gs).T
    b = x @ dequantize_rows(uq, us).T
    return a / (1.0 + np.exp(-a)) * b


def down_fp8(hq: np.ndarray, hs: np.ndarray, dq: np.ndarray, ds: np.ndarray) -> np.ndarray:
    """o = (s_h q_h)(s_d q_d)^T in float64: hq [n, f] codes with row scales hs [n]; dq [d, f] the
    codes of one expert's W_down rows (one per output channel) with scales ds [d]."""
    return dequantize_rows(hq, hs) @ dequantize_rows(dq, ds).T


def quantize_expert_rows(W: np.ndarray):
    """Row quantisation of every expert's matrix: W [G, rows, cols] (exact fp32 values) ->
    codes [G, rows, cols] uint8 and scales [G, rows] float32."""
    W = np.asarray(W, dtype=np.float32)
    codes = np.empty(W.shape, np.uint8)
    scales = np.empty(W.shape[:2], np.float32)
    for g in range(W.shape[0]):
        codes[g], scales[g] = quantize_rows_e4m3(W[g])
    return codes, scales


def expert_forward_fp8(xr: np.ndarray, gq, gs, uq, us, dq, ds) -> np.ndarray:
    """One expert's output rows with e4m3 GEMMs, in the order the forward takes the steps: the x
    rows are quantised per row, h = silu(a) * b from gate_up_fp8, h is held in bf16 (rounded once,
    nearest even) and quantised per row, and o = down_fp8 of those codes.  xr [n, d] exact values."""
    xq, xsc = quantize_rows_e4m3(np.asarray(xr, np.float32))
    h = gate_up_fp8(xq, xsc, gq, gs, uq, us)
    hq, hsc = quantize_rows_e4m3(f64_to_bf16_value(h).astype(np.float32))
    return down_fp8(hq, hsc, dq, ds)


def layer_forward_fp8(L) -> np.ndarray:
    """y [T, d] (float64) of a Layer whose expert weights are quantised per row (W_gate and W_up
    rows: channels of d_ff; W_down rows: channels of d_model): routing, dispatch and combine as
    Layer.forward, every expert's SwiGLU FFN through expert_forward_fp8."""
    R, D = L.routing(), L.dispatch()
    T, k, d = L.T, L.k, L.d
    gq, gs = quantize_expert_rows(as_f64(L.inp["W_gate"]))
    uq, us = quantize_expert_rows(as_f64(L.inp["W_up"]))
    dq, ds = quantize_expert_rows(as_f64(L.inp["W_down"]))

    def expert(g, xr):
        return expert_forward_fp8(xr, gq[g], gs[g], uq[g], us[g], dq[g], ds[g])

    o_slot = np.zeros((T, k, d))
    for e in range(L.E):
        rows = np.arange(D.offsets[e], D.offsets[e + 1])
        if rows.size == 0:
            continue
        slots = D.slot_of_row[rows]
        o_slot[slots // k, slots % k] = expert(e, L.x[slots // k])
    shared = [expert(L.E + s, L.x) for s in range(L.S)]
    return combine(o_slot, R.gates, D.row_of_slot >= 0, shared)


def token_outputs_fp8(L, tokens: np.ndarray, cols: np.ndarray) -> np.ndarray:
    """y[tokens][:, cols] of the e4m3 forward, one token at a time (for full-size workloads).

    Routing as Layer.token_outputs (the capacity, when set, needs the queues over all tokens).  Only
    the experts the tokens visit are quantised, and of W_down only the rows of the requested output
    channels: each row's quantisation depends on that row alone."""
    tokens = np.asarray(tokens, np.int64)
    cols = np.asarray(cols, np.int64)
    R = L.routing()
    idx, g = R.idx[tokens], R.gates[tokens]
    kept = L.dispatch().row_of_slot[tokens] >= 0 if L.C is not None else np.ones(idx.shape, bool)
    xs = L.x[tokens]
    y = np.zeros((tokens.size, cols.size))
    for e in range(L.E + L.S):
        if e < L.E:
            sel = np.argwhere((idx == e) & kept)
            if sel.size == 0:
                continue
            ti, gw = sel[:, 0], g[sel[:, 0], sel[:, 1]]
        else:
            ti, gw = np.arange(tokens.size), np.ones(tokens.size)
        gq, gs = quantize_rows_e4m3(as_f64(L.inp["W_gate"][e]).astype(np.float32))
        uq, us = quantize_rows_e4m3(as_f64(L.inp["W_up"][e]).astype(np.float32))
        dq, ds = quantize_rows_e4m3(as_f64(L.inp["W_down"][e][cols]).astype(np.float32))
        o = expert_forward_fp8(xs[ti], gq, gs, uq, us, dq, ds)
        np.add.at(y, ti, gw[:, None] * o)
    return y


# ---------------------------------------------------------------------------------------------
# e4m3 backward (moe_layer_bwd_fp8 computes it)
#
# Reading, continuing the forward's: the two data-gradient products take e4m3 operands,
#   dh' = dY W_d        left: dY rows, per row;  right: the rows of W_d^T (W_d's columns, one
#                       scale per d_ff channel)
#   dX  = dA W_g + dB W_u   left: the row [dA | dB], one scale over both halves; right: the rows of
#                       [W_g^T | W_u^T] (column i of W_g and of W_u, one scale per d_model channel)
# a and b come from the forward's codes; dh', dA, dB and Hg are held in bf16 (the precision of
# those buffers in the bf16 path) and quantised from those bf16 values; the weight gradients stay
# bf16 GEMMs (their K runs over rows), so they take the rounded dA, dB, Hg exactly.
# ---------------------------------------------------------------------------------------------

def quantize_cols_e4m3(W: np.ndarray):
    """Per-column e4m3 codes of a [rows, cols] matrix of exact fp32 values, returned as the codes
    of W^T ([cols, rows], the K-major operand whose rows are W's columns) and one scale per column."""
    return quantize_rows_e4m3(np.asarray(W, np.float32).T)


def gate_up_pre_fp8(xq, xs, gq, gs, uq, us):
    """a and b (float64) of quantised rows, before the SwiGLU: the products gate_up_fp8 combines."""
    x = dequantize_rows(xq, xs)
    return x @ dequantize_rows(gq, gs).T, x @ dequantize_rows(uq, us).T


def dh_fp8(dyq, dys, wdtq, wdts):
    """dh' = (s_dy q_dy)(s_w q_w)^T: dY rows [n, d] codes with row scales; wdtq [f, d] the codes of
    W_d^T (W_d's columns) with one scale per d_ff channel."""
    return dequantize_rows(dyq, dys) @ dequantize_rows(wdtq, wdts).T


def dx_fp8(dabq, dabs, wgutq, wguts):
    """dX = [dA | dB] [W_g ; W_u]: dabq [n, 2f] codes of the joined rows with their scales; wgutq
    [d, 2f] the codes of [W_g^T | W_u^T] (column i of W_g then of W_u) with one scale per d_model
    channel."""
    return dequantize_rows(dabq, dabs) @ dequantize_rows(wgutq, wguts).T


def _bf16(v):
    return f64_to_bf16_value(v)


def expert_backward_fp8(xr, dyr, g, Wg, Wu, Wd):
    """The e4m3 backward of g * expert(xr) for rows xr (exact fp32 values) with upstream dyr and
    per-row gate g, in the steps and precisions of the reading above.

    Returns dxr, dWg, dWu, dWd, dg as expert_backward does."""
    f32 = lambda v: np.asarray(v, np.float32)
    xq, xs = quantize_rows_e4m3(f32(xr))
    gq, gs = quantize_rows_e4m3(f32(Wg))
    uq, us = quantize_rows_e4m3(f32(Wu))
    a, b = gate_up_pre_fp8(xq, xs, gq, gs, uq, us)
    dyq, dys = quantize_rows_e4m3(f32(dyr))
    wdtq, wdts = quantize_cols_e4m3(f32(Wd))
    dhp = _bf16(dh_fp8(dyq, dys, wdtq, wdts))             # dh' held in bf16
    s = 1.0 / (1.0 + np.exp(-a))
    h = a * s * b
    dg = np.sum(dhp * h, axis=1)
    dh = np.asarray(g, np.float64)[:, None] * dhp
    dA = _bf16(dh * b * s * (1.0 + a * (1.0 - s)))
    dB = _bf16(dh * (a * s))
    Hg = _bf16(np.asarray(g, np.float64)[:, None] * h)
    dabq, dabs = quantize_rows_e4m3(f32(np.concatenate([dA, dB], axis=1)))
    wgutq, wguts = quantize_cols_e4m3(f32(np.concatenate([Wg, Wu], axis=0)))
    dxr = dx_fp8(dabq, dabs, wgutq, wguts)
    xr64 = np.asarray(xr, np.float64)
    dWg = dA.T @ xr64
    dWu = dB.T @ xr64
    dWd = np.asarray(dyr, np.float64).T @ Hg
    return dxr, dWg, dWu, dWd, dg


def layer_backward_fp8(L) -> dict:
    """All gradients of sum(dy * y) with the e4m3 backward of every expert (routing, dispatch and the
    router backward as Layer.backward)."""
    R, D = L.routing(), L.dispatch()
    T, k, d, f, E, S = L.T, L.k, L.d, L.f, L.E, L.S
    dx = np.zeros((T, d))
    dW_gate, dW_up, dW_down = np.zeros((E + S, f, d)), np.zeros((E + S, f, d)), np.zeros((E + S, d, f))
    dgates = np.zeros((T, k))
    for e in range(E + S):
        Wg, Wu, Wd = L.W(e)
        if e < E:
            rows = np.arange(D.offsets[e], D.offsets[e + 1])
            if rows.size == 0:
                continue
            slots = D.slot_of_row[rows]
            t_of, j_of = slots // k, slots % k
            gw = R.gates[t_of, j_of]
        else:
            t_of, j_of, gw = np.arange(T), None, np.ones(T)
        dxr, dWg, dWu, dWd, dg = expert_backward_fp8(L.x[t_of], L.dy[t_of], gw, Wg, Wu, Wd)
        np.add.at(dx, t_of, dxr)
        dW_gate[e], dW_up[e], dW_down[e] = dWg, dWu, dWd
        if j_of is not None:
            dgates[t_of, j_of] = dg
    dl = router_backward_logits(R.p, R.idx, R.gates, dgates, L.renorm)
    dW_r, db_r, dx_r = router_backward(L.x, L.inp["W_r"], dl)
    return dict(dx=dx + dx_r, dW_r=dW_r, db_r=db_r, dW_gate=dW_gate, dW_up=dW_up, dW_down=dW_down,
                dgates=dgates, dlogits=dl)


def token_grads_fp8(L, tokens: np.ndarray) -> dict:
    """dx[tokens] and dgates[tokens] of the e4m3 backward, token by token (for full-size workloads).

    A token's rows go through expert_backward_fp8 on their own: the quantisation of an x, dY or
    [dA | dB] row depends on that row alone, and each expert's weights are quantised whole (their
    column scales span the expert).  The router term follows from the token's own routing and gate
    gradients.  Routing as Layer.token_outputs (a capacity needs the queues over all tokens)."""
    from .moe_oracle import gates_of, router_logits, softmax, topk_by_rank
    tokens = np.asarray(tokens, np.int64)
    k = L.k
    if L.C is not None:
        R = L.routing()
        p, idx, g = R.p[tokens], R.idx[tokens], R.gates[tokens]
        kept = L.dispatch().row_of_slot[tokens] >= 0
    else:
        lg = router_logits(L.x[tokens], L.inp["W_r"], L.inp.get("b_r"))
        p = softmax(lg)
        idx = topk_by_rank(lg, k)
        g = gates_of(p, idx, L.renorm)
        kept = np.ones(idx.shape, dtype=bool)
    n = tokens.size
    xs, dys = L.x[tokens], L.dy[tokens]
    dx = np.zeros((n, L.d))
    dgates = np.zeros((n, k))
    for e in range(L.E + L.S):
        if e < L.E:
            sel = np.argwhere((idx == e) & kept)
            if sel.size == 0:
                continue
            ti, jj = sel[:, 0], sel[:, 1]
            gw = g[ti, jj]
        else:
            ti, jj, gw = np.arange(n), None, np.ones(n)
        Wg, Wu, Wd = L.W(e)
        dxr, _, _, _, dg = expert_backward_fp8(xs[ti], dys[ti], gw, Wg, Wu, Wd)
        np.add.at(dx, ti, dxr)
        if jj is not None:
            dgates[ti, jj] = dg
    dl = router_backward_logits(p, idx, g, dgates, L.renorm)
    dx += dl @ np.asarray(L.inp["W_r"], np.float64).T
    return dict(dx=dx, dgates=dgates)


def weight_grad_columns_fp8(L, e: int, cols: np.ndarray) -> dict:
    """dW_gate[e][cols, :], dW_up[e][cols, :] and dW_down[e][:, cols] of the e4m3 backward.

    Hidden unit c needs only column c of a, b and dh' over the expert's rows: a and b from row c of
    W_gate and W_up (each quantised with its own scale), dh' from column c of W_down (its own
    scale), the x and dY rows quantised per row -- expert_backward_fp8's steps, for these units."""
    cols = np.asarray(cols, np.int64)
    k = L.k
    if e < L.E:
        D, R = L.dispatch(), L.routing()
        rows = np.arange(D.offsets[e], D.offsets[e + 1])
        slots = D.slot_of_row[rows]
        t_of, j_of = slots // k, slots % k
        gw = R.gates[t_of, j_of]
    else:
        t_of = np.arange(L.T)
        gw = np.ones(L.T)
    f32 = lambda v: np.asarray(v, np.float32)
    Wg, Wu, Wd = L.W(e)
    xr, dyr = L.x[t_of], L.dy[t_of]
    xq, xs = quantize_rows_e4m3(f32(xr))
    gq, gs = quantize_rows_e4m3(f32(Wg[cols]))
    uq, us = quantize_rows_e4m3(f32(Wu[cols]))
    a, b = gate_up_pre_fp8(xq, xs, gq, gs, uq, us)
    dyq, dys = quantize_rows_e4m3(f32(dyr))
    wdtq, wdts = quantize_cols_e4m3(f32(Wd[:, cols]))
    dhp = _bf16(dh_fp8(dyq, dys, wdtq, wdts))
    s = 1.0 / (1.0 + np.exp(-a))
    h = a * s * b
    dh = gw[:, None] * dhp
    dA = _bf16(dh * b * s * (1.0 + a * (1.0 - s)))
    dB = _bf16(dh * (a * s))
    Hg = _bf16(gw[:, None] * h)
    return dict(dW_gate=dA.T @ xr, dW_up=dB.T @ xr, dW_down=dyr.T @ Hg)


# ---------------------------------------------------------------------------------------------
# MXFP8 (oracle only: block-scaled e4m3 as the kind::mxf8f6f4 MMAs consume it; not built yet)
#
# Reading (OCP Microscaling Formats v1.0, conversion of a block): every 32 consecutive values
# along K share one power-of-two scale X = 2^(floor(log2(amax)) - 8), 8 being the exponent of the
# largest normal E4M3 value (448 = 1.75 * 2^8); each element is RNE(v / X) in E4M3, saturated to
# +-448 (amax / X lies in [256, 512), so the top of a block can saturate); X is stored as an E8M0
# byte (exponent + 127).  An all-zero block takes the smallest scale, 2^-127 (byte 0).
# ---------------------------------------------------------------------------------------------

MX_BLOCK = 32
_E4M3_EMAX = 8


def mx_quantize_e4m3(rows: np.ndarray):
    """MX E4M3 codes of a [n, width] array of exact fp32 values, width a multiple of 32: returns
    (codes uint8 [n, width], scale exponents int [n, width / 32]).  The block's scale is
    2^exponent; the E8M0 byte is exponent + 127."""
    v = np.asarray(rows, np.float64)
    n, w = v.shape
    assert w % MX_BLOCK == 0
    blocks = v.reshape(n, w // MX_BLOCK, MX_BLOCK)
    amax = np.abs(blocks).max(axis=2)
    with np.errstate(divide="ignore"):
        e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - _E4M3_EMAX, -127)
    e = np.clip(e, -127, 127).astype(np.int64)
    scaled = blocks / np.ldexp(1.0, e)[:, :, None]         # exact: a power-of-two division
    return e4m3_encode_rne(scaled).reshape(n, w), e


def mx_dequantize(codes: np.ndarray, exps: np.ndarray) -> np.ndarray:
    """float64 values of MX E4M3 rows: each code's value times its block's 2^exponent (exact)."""
    c = np.asarray(codes)
    n, w = c.shape
    vals = e4m3_decode(c).reshape(n, w // MX_BLOCK, MX_BLOCK)
    return (vals * np.ldexp(1.0, np.asarray(exps, np.int64))[:, :, None]).reshape(n, w)


def mx_matmul(aq, ae, bq, be) -> np.ndarray:
    """A B^T in float64 from MX operands both blocked along K: aq [m, K], bq [n, K] codes with their
    per-block exponents."""
    return mx_dequantize(aq, ae) @ mx_dequantize(bq, be).T
