"""Parity of each C-ABI step with the fp64 oracle on the same seeded inputs (GPU).

Assignments flow from the oracle into the GPU calls (moe_dispatch takes idx as an input), never
the other way, so every downstream check is "given identical assignments".  Inputs a step needs
that the oracle does not produce (expert outputs for the combine, gate gradients for the router
backward, row gradients for the input combine) are seeded synthetic tensors.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from cases import CASES, case
from harness import (check_close, check_routing, check_weight_grad, from_dev, from_dev_bf16,
                     segment_rows, to_dev, to_dev_bf16)

pytestmark = pytest.mark.gpu

ALL = list(CASES)


def _cfg(moe, c):
    return moe.config_from(c)


def _dispatch(moe, c, inp, L):
    """Run moe_dispatch on the oracle's assignments; return device tensors and the buffers."""
    mc = _cfg(moe, c)
    buf = moe.Buffers.allocate(mc)
    T, k, E, d = c["T"], c["k"], c["E"], c["d"]
    idx = to_dev(L.routing().idx.astype(np.int32))
    x = to_dev_bf16(inp["x"])
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    row_of_slot = torch.empty(T * k, dtype=torch.int32, device="cuda")
    token_of_row = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    x_perm = torch.full((buf.rows, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch(mc, idx, x, counts, offsets, row_of_slot, token_of_row, x_perm, buf.ws)
    assert moe.moe_check_error(buf.ws) == 0
    return mc, buf, dict(idx=idx, x=x, counts=counts, offsets=offsets, row_of_slot=row_of_slot,
                         token_of_row=token_of_row, x_perm=x_perm)


@pytest.mark.parametrize("name", ALL)
def test_route(moe, name):
    c, inp, L = case(name)
    mc = _cfg(moe, c)
    T, k, E = c["T"], c["k"], c["E"]
    x = to_dev_bf16(inp["x"])
    W_r = to_dev(inp["W_r"])
    b_r = to_dev(inp["b_r"]) if inp["b_r"] is not None else None
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    gates = torch.empty(T, k, dtype=torch.float32, device="cuda")
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    buf = moe.Buffers.allocate(mc)
    moe.moe_route(mc, x, W_r, b_r, idx, gates, logits, buf.ws)
    assert moe.moe_check_error(buf.ws) == 0
    torch.cuda.synchronize()
    R = L.routing()
    lg = from_dev(logits).astype(np.float64)
    assert np.max(np.abs(lg - R.logits) / (1.0 + np.abs(R.logits))) < 2e-5
    same = check_routing(from_dev(idx), from_dev(gates), R, k)
    assert same.mean() > 0.99


@pytest.mark.parametrize("name", ALL)
def test_dispatch(moe, name):
    c, inp, L = case(name)
    mc, buf, t = _dispatch(moe, c, inp, L)
    D = L.dispatch()
    T, k, S = c["T"], c["k"], c["S"]
    assert np.array_equal(from_dev(t["counts"]), D.counts)
    assert from_dev(t["counts"]).sum() == T * k
    assert np.array_equal(from_dev(t["offsets"]), D.offsets)
    assert np.array_equal(from_dev(t["row_of_slot"]).reshape(T, k), D.row_of_slot)
    n = int(D.offsets[-1])
    tor = from_dev(t["token_of_row"])
    assert np.array_equal(tor[:n], D.token_of_row)
    assert np.all(tor[n:] == -7), "entries past the kept rows must be left untouched"
    # x_perm follows the documented padded layout exactly (a pure copy: bit-exact)
    kept, P = segment_rows(D, T, S)
    xp = from_dev_bf16(t["x_perm"])
    x = oracle.bf16_to_f64(inp["x"])
    for g in range(len(kept)):
        rows = xp[P[g]:P[g] + kept[g]]
        ref = x[D.token_of_row[D.offsets[g]:D.offsets[g + 1]]] if g < c["E"] else x
        assert np.array_equal(rows, ref), f"segment {g}"
        assert np.all(xp[P[g] + kept[g]:P[g + 1]] == 0), f"pad rows of segment {g}"


@pytest.mark.parametrize("name", ALL)
def test_expert_ffn_fwd(moe, name):
    c, inp, L = case(name)
    mc, buf, t = _dispatch(moe, c, inp, L)
    D = L.dispatch()
    T, S, E, d = c["T"], c["S"], c["E"], c["d"]
    Wg, Wu, Wd = (to_dev_bf16(inp[n]) for n in ("W_gate", "W_up", "W_down"))
    o_perm = torch.full((buf.rows, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn_fwd(mc, t["x_perm"], Wg, Wu, Wd, o_perm, buf.ws)
    assert moe.moe_check_error(buf.ws) == 0
    kept, P = segment_rows(D, T, S)
    op = from_dev_bf16(o_perm)
    refs, gots = [], []
    for g in range(E + S):
        if kept[g] == 0:
            continue
        toks = D.token_of_row[D.offsets[g]:D.offsets[g + 1]] if g < E else np.arange(T)
        refs.append(oracle.expert_forward(L.x[toks], *L.W(g))[3])
        gots.append(op[P[g]:P[g] + kept[g]])
        assert np.all(op[P[g] + kept[g]:P[g + 1]] == 0), f"pad rows of segment {g}"
    check_close("o_perm", np.concatenate(gots), np.concatenate(refs))


@pytest.mark.parametrize("name", ALL)
def test_combine(moe, name):
    c, inp, L = case(name)
    mc, buf, t = _dispatch(moe, c, inp, L)
    D, R = L.dispatch(), L.routing()
    T, k, S, E, d = c["T"], c["k"], c["S"], c["E"], c["d"]
    kept, P = segment_rows(D, T, S)
    o_bits = synth.normal_bf16(7, "aux", (buf.rows, d), 1.0, chunk=3)
    o = oracle.bf16_to_f64(o_bits)
    gates32 = R.gates.astype(np.float32)
    # oracle: slot (t, j) of expert e reads row P_e + position (the documented layout)
    o_slot = np.zeros((T, k, d))
    live = D.row_of_slot >= 0
    for tt, j in zip(*np.nonzero(live)):
        e = R.idx[tt, j]
        o_slot[tt, j] = o[P[e] + D.position[tt, j]]
    shared = [o[P[E + s]:P[E + s] + T] for s in range(S)]
    y_ref = oracle.combine(o_slot, gates32.astype(np.float64), live, shared)
    y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(mc, to_dev_bf16(o_bits), to_dev(gates32), y, buf.ws)
    assert moe.moe_check_error(buf.ws) == 0
    check_close("y", from_dev_bf16(y), y_ref)


@pytest.mark.parametrize("name", ALL)
def test_expert_ffn_bwd(moe, name):
    c, inp, L = case(name)
    mc, buf, t = _dispatch(moe, c, inp, L)
    D, R = L.dispatch(), L.routing()
    T, k, S, E, d, f = c["T"], c["k"], c["S"], c["E"], c["d"], c["f"]
    G = E + S
    Wg, Wu, Wd = (to_dev_bf16(inp[n]) for n in ("W_gate", "W_up", "W_down"))
    gates32 = R.gates.astype(np.float32)
    dx_perm = torch.full((buf.rows, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    dgates = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    dWg = torch.full((G, f, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    dWu = torch.full_like(dWg, float("nan"))
    dWd = torch.full((G, d, f), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn_bwd(mc, t["x_perm"], to_dev_bf16(inp["dy"]), to_dev(gates32), Wg, Wu, Wd,
                           dx_perm, dgates, dWg, dWu, dWd, buf.ws)
    assert moe.moe_check_error(buf.ws) == 0
    kept, P = segment_rows(D, T, S)
    dxp = from_dev_bf16(dx_perm)
    ref_dx, got_dx = [], []
    ref_dg = np.zeros((T, k))
    ref_W = [np.zeros((G, f, d)), np.zeros((G, f, d)), np.zeros((G, d, f))]
    for g in range(G):
        if kept[g] == 0:
            continue
        if g < E:
            slots = D.slot_of_row[D.offsets[g]:D.offsets[g + 1]]
            toks, js = slots // k, slots % k
            gw = gates32[toks, js].astype(np.float64)
        else:
            toks, gw = np.arange(T), np.ones(T)
        dxr, dWg_r, dWu_r, dWd_r, dg = oracle.expert_backward(L.x[toks], L.dy[toks], gw, *L.W(g))
        ref_dx.append(dxr)
        got_dx.append(dxp[P[g]:P[g] + kept[g]])
        ref_W[0][g], ref_W[1][g], ref_W[2][g] = dWg_r, dWu_r, dWd_r
        if g < E:
            ref_dg[toks, js] = dg
        assert np.all(dxp[P[g] + kept[g]:P[g + 1]] == 0), f"pad rows of segment {g}"
    check_close("dx_perm", np.concatenate(got_dx), np.concatenate(ref_dx))
    check_close("dgates", from_dev(dgates), ref_dg)
    check_weight_grad("dW_gate", from_dev_bf16(dWg), ref_W[0])
    check_weight_grad("dW_up", from_dev_bf16(dWu), ref_W[1])
    check_weight_grad("dW_down", from_dev_bf16(dWd), ref_W[2])


@pytest.mark.parametrize("name", ALL)
def test_router_bwd(moe, name):
    c, inp, L = case(name)
    mc = _cfg(moe, c)
    buf = moe.Buffers.allocate(mc)
    R = L.routing()
    T, k, E, d = c["T"], c["k"], c["E"], c["d"]
    gates32 = R.gates.astype(np.float32)
    dg32 = synth.normal_f32(11, "aux", (T, k), 1.0, chunk=5)
    dl_ref = oracle.router_backward_logits(R.p, R.idx, gates32.astype(np.float64),
                                           dg32.astype(np.float64), bool(c["renorm"]))
    dWr_ref, db_ref, _ = oracle.router_backward(L.x, inp["W_r"], dl_ref)
    dlogits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    dW_r = torch.empty(d, E, dtype=torch.float32, device="cuda")
    db_r = torch.empty(E, dtype=torch.float32, device="cuda")
    b_r = to_dev(inp["b_r"]) if inp["b_r"] is not None else None
    moe.moe_router_bwd(mc, to_dev_bf16(inp["x"]), to_dev(inp["W_r"]), b_r, to_dev(R.idx.astype(np.int32)),
                       to_dev(gates32), to_dev(dg32), dlogits, dW_r, db_r, buf.ws)
    assert moe.moe_check_error(buf.ws) == 0
    check_close("dlogits", from_dev(dlogits), dl_ref)
    check_close("dW_r", from_dev(dW_r), dWr_ref)
    check_close("db_r", from_dev(db_r), db_ref)


@pytest.mark.parametrize("name", ALL)
@pytest.mark.parametrize("with_router", [True, False])
def test_combine_bwd(moe, name, with_router):
    c, inp, L = case(name)
    mc, buf, t = _dispatch(moe, c, inp, L)
    D, R = L.dispatch(), L.routing()
    T, k, S, E, d = c["T"], c["k"], c["S"], c["E"], c["d"]
    kept, P = segment_rows(D, T, S)
    g_bits = synth.normal_bf16(9, "aux", (buf.rows, d), 1.0, chunk=7)
    grows = oracle.bf16_to_f64(g_bits)
    dl = synth.normal_f32(9, "aux", (T, E), 0.1, chunk=8)
    ref = np.zeros((T, d))
    for tt, j in zip(*np.nonzero(D.row_of_slot >= 0)):
        ref[tt] += grows[P[R.idx[tt, j]] + D.position[tt, j]]
    for s in range(S):
        ref += grows[P[E + s]:P[E + s] + T]
    if with_router:
        ref += dl.astype(np.float64) @ np.asarray(inp["W_r"], np.float64).T
    dx = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    moe.moe_combine_bwd(mc, to_dev_bf16(g_bits), to_dev(dl) if with_router else None,
                        to_dev(inp["W_r"]) if with_router else None, dx, buf.ws)
    assert moe.moe_check_error(buf.ws) == 0
    check_close("dx", from_dev_bf16(dx), ref)
