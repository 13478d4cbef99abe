"""Degenerate and boundary cases through the step calls (GPU): experts with no rows, one expert
taking every token, a single token, widths that are multiples of 64 but not of 128 (the GPT-OSS
width 2880), and the largest capacity drop (C = 1)."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from harness import (check_close, check_weight_grad, from_dev, from_dev_bf16, padded_starts, to_dev,
                     to_dev_bf16)

pytestmark = pytest.mark.gpu


def _inputs(T, d, f, E, S, seed):
    G = E + S
    return dict(x=synth.normal_bf16(seed, "x", (T, d), 1.0),
                W_gate=synth.normal_bf16(seed, "W_gate", (G, f, d), 1 / math.sqrt(d)),
                W_up=synth.normal_bf16(seed, "W_up", (G, f, d), 1 / math.sqrt(d)),
                W_down=synth.normal_bf16(seed, "W_down", (G, d, f), 1 / math.sqrt(f)),
                dy=synth.normal_bf16(seed, "dy", (T, d), 1.0))


def run_steps(moe, T, d, f, E, k, S, idx, gates, cf=0.0, seed=0):
    """dispatch -> expert fwd -> combine, and expert bwd, on given assignments; check all against
    the oracle's definitions on the same assignments."""
    inp = _inputs(T, d, f, E, S, seed)
    mc = moe.config(T=T, d=d, f=f, E=E, k=k, S=S, cf=cf)
    buf = moe.Buffers.allocate(mc)
    G = E + S
    C = oracle.capacity_of(T, k, E, cf)
    D = oracle.dispatch(idx, E, C)
    kept = np.concatenate([D.kept, np.full(S, T)])
    P = padded_starts(kept)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    ros = torch.empty(T * k, dtype=torch.int32, device="cuda")
    tor = torch.empty(T * k, dtype=torch.int32, device="cuda")
    x_perm = torch.empty(buf.rows, d, dtype=torch.bfloat16, device="cuda")
    o_perm = torch.empty_like(x_perm)
    dx_perm = torch.empty_like(x_perm)
    Wg, Wu, Wd = (to_dev_bf16(inp[n]) for n in ("W_gate", "W_up", "W_down"))
    g_dev = to_dev(gates.astype(np.float32))
    moe.moe_dispatch(mc, to_dev(idx.astype(np.int32)), to_dev_bf16(inp["x"]), counts, offsets, ros, tor,
                     x_perm, buf.ws)
    moe.moe_expert_ffn_fwd(mc, x_perm, Wg, Wu, Wd, o_perm, buf.ws)
    y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(mc, o_perm, g_dev, y, buf.ws)
    dgates = torch.empty(T, k, dtype=torch.float32, device="cuda")
    dWg, dWu = torch.empty_like(Wg), torch.empty_like(Wu)
    dWd = torch.empty_like(Wd)
    moe.moe_expert_ffn_bwd(mc, x_perm, to_dev_bf16(inp["dy"]), g_dev, Wg, Wu, Wd, dx_perm, dgates,
                           dWg, dWu, dWd, buf.ws)
    assert moe.moe_check_error(buf.ws) == 0
    assert np.array_equal(from_dev(counts), D.counts)
    assert np.array_equal(from_dev(offsets), D.offsets)
    assert np.array_equal(from_dev(ros).reshape(T, k), D.row_of_slot)

    x = oracle.bf16_to_f64(inp["x"])
    dy = oracle.bf16_to_f64(inp["dy"])
    g64 = gates.astype(np.float32).astype(np.float64)
    o_slot = np.zeros((T, k, d))
    y_shared = []
    ref_W = [np.zeros((G, f, d)), np.zeros((G, f, d)), np.zeros((G, d, f))]
    ref_dg = np.zeros((T, k))
    ref_dxp, got_dxp = [], []
    for g in range(G):
        W = tuple(oracle.bf16_to_f64(inp[n][g]) for n in ("W_gate", "W_up", "W_down"))
        if g < E:
            slots = D.slot_of_row[D.offsets[g]:D.offsets[g + 1]]
            toks, js = slots // k, slots % k
            gw = g64[toks, js]
        else:
            toks, js, gw = np.arange(T), None, np.ones(T)
        if toks.size == 0:
            continue
        o = oracle.expert_forward(x[toks], *W)[3]
        dxr, a, b, c, dg = oracle.expert_backward(x[toks], dy[toks], gw, *W)
        ref_W[0][g], ref_W[1][g], ref_W[2][g] = a, b, c
        ref_dxp.append(dxr)
        got_dxp.append(from_dev_bf16(dx_perm[P[g]:P[g] + kept[g]]))   # rows past kept hold no values
        if g < E:
            o_slot[toks, js] = o
            ref_dg[toks, js] = dg
        else:
            y_shared.append(o)
    y_ref = oracle.combine(o_slot, g64, D.row_of_slot >= 0, y_shared)
    check_close("y", from_dev_bf16(y), y_ref)
    check_close("dgates", from_dev(dgates), ref_dg)
    check_close("dx_perm", np.concatenate(got_dxp), np.concatenate(ref_dxp))
    check_weight_grad("dW_gate", from_dev_bf16(dWg), ref_W[0])
    check_weight_grad("dW_up", from_dev_bf16(dWu), ref_W[1])
    check_weight_grad("dW_down", from_dev_bf16(dWd), ref_W[2])


def test_all_tokens_to_one_expert(moe):
    T, E, k = 300, 8, 1
    idx = np.zeros((T, k), dtype=np.int32)           # experts 1..7 get no rows
    run_steps(moe, T, 128, 128, E, k, 0, idx, np.full((T, k), 0.7))


def test_one_expert_in_every_token_plus_empty_experts(moe):
    T, E, k = 257, 16, 2
    rng = np.random.default_rng(1)
    idx = np.stack([np.zeros(T, np.int32), rng.integers(1, 4, T).astype(np.int32)], 1)
    run_steps(moe, T, 192, 128, E, k, 0, idx, rng.random((T, k)))


def test_single_token(moe):
    idx = np.array([[3, 1]], dtype=np.int32)
    run_steps(moe, 1, 64, 64, 4, 2, 1, idx, np.array([[0.6, 0.3]]))


def test_gptoss_width(moe):
    T, E, k = 160, 4, 2
    idx = synth.random_assignments(5, T, E, k)
    run_steps(moe, T, 2880, 192, E, k, 0, idx, np.full((T, k), 0.5))


def test_gptoss_ffn_width(moe):
    T, E, k = 150, 4, 2
    idx = synth.random_assignments(6, T, E, k)
    run_steps(moe, T, 192, 2880, E, k, 0, idx, np.full((T, k), 0.5))


def test_many_tokens_per_warp_ragged_width(moe):
    # more tokens than gather warps (each warp owns several tokens) and rows of 40 16-byte vectors
    T, E, k = 24000, 8, 2
    idx = synth.random_assignments(8, T, E, k)
    run_steps(moe, T, 320, 64, E, k, 1, idx, np.full((T, k), 0.5))


def test_capacity_one(moe):
    T, E, k = 200, 8, 2
    idx = synth.random_assignments(7, T, E, k, skew=1.5)
    cf = 1.0 / (T * k / E)                           # ceil(cf*T*k/E) = 1: one row per expert
    run_steps(moe, T, 128, 128, E, k, 0, idx, np.full((T, k), 0.5), cf=cf)
