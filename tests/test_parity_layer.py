"""Parity of the fused moe_layer_fwd / moe_layer_bwd calls with the fp64 oracle (GPU)."""
import numpy as np
import pytest
import torch

from cases import CASES, case
from harness import (check_close, check_gates, check_routing, check_weight_grad, decided_tokens,
                     from_dev, from_dev_bf16, to_dev, to_dev_bf16)

pytestmark = pytest.mark.gpu


def run_layer(moe, c, inp, buf=None):
    mc = moe.config_from(c)
    buf = buf or moe.Buffers.allocate(mc)
    T, d, f, E, S = c["T"], c["d"], c["f"], c["E"], c["S"]
    G = E + S
    dev = dict(x=to_dev_bf16(inp["x"]), W_r=to_dev(inp["W_r"]),
               b_r=to_dev(inp["b_r"]) if inp["b_r"] is not None else None,
               Wg=to_dev_bf16(inp["W_gate"]), Wu=to_dev_bf16(inp["W_up"]), Wd=to_dev_bf16(inp["W_down"]),
               dy=to_dev_bf16(inp["dy"]))
    y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    moe.moe_layer_fwd(mc, dev["x"], dev["W_r"], dev["b_r"], dev["Wg"], dev["Wu"], dev["Wd"], y, buf.saved, buf.ws)
    out = dict(y=y, dx=torch.empty(T, d, dtype=torch.bfloat16, device="cuda"),
               dW_r=torch.empty(d, E, dtype=torch.float32, device="cuda"),
               db_r=torch.empty(E, dtype=torch.float32, device="cuda"),
               dWg=torch.empty(G, f, d, dtype=torch.bfloat16, device="cuda"),
               dWu=torch.empty(G, f, d, dtype=torch.bfloat16, device="cuda"),
               dWd=torch.empty(G, d, f, dtype=torch.bfloat16, device="cuda"))
    moe.moe_layer_bwd(mc, dev["x"], dev["W_r"], dev["b_r"], dev["Wg"], dev["Wu"], dev["Wd"], buf.saved,
                      dev["dy"], out["dx"], out["dW_r"], out["db_r"], out["dWg"], out["dWu"], out["dWd"], buf.ws)
    status = moe.moe_check_error(buf.ws)
    assert status == 0, moe.moe_status_string(status)
    k = c["k"]
    sv = buf.saved.view(torch.int32)
    out["idx"] = sv[:T * k].view(T, k)
    out["gates"] = buf.saved.view(torch.float32)[T * k:2 * T * k].view(T, k)
    return out, buf


@pytest.mark.parametrize("name", list(CASES))
def test_layer_fwd_bwd(moe, name):
    c, inp, L = case(name)
    out, buf = run_layer(moe, c, inp)
    check_layer(moe, c, inp, L, out, buf)


# Kept activations: the forward stores a, b of the leading expert-ordered rows and the backward
# uses them instead of recomputing (all rows, or a prefix that ends inside a segment).
@pytest.mark.parametrize("name,keep", [("ragged_mixtral", -1), ("ragged_mixtral", 256), ("deepseek_small", -1),
                                       ("deepseek_small", 768), ("gptoss_small", 512), ("qwen_small", -1),
                                       ("router_e96_k8", 256), ("tiny", 100)])
def test_layer_kept_activations(moe, name, keep):
    c, inp, L = case(name)
    c = dict(c)
    c["keep_rows"] = moe.moe_perm_rows(moe.config_from(c)) if keep < 0 else keep
    out, buf = run_layer(moe, c, inp)
    check_layer(moe, c, inp, L, out, buf)


def check_layer(moe, c, inp, L, out, buf):
    """The forward where it is unique and every gradient under identical assignments.

    Top-k is checked by the routing rule.  y of a token depends only on the assignments queued
    before it (its own, and with a capacity those of earlier tokens), so it is compared on the
    tokens whose routing agrees (with a capacity: before the first difference).  The gradients
    depend on every token's assignment: when a near-tie went the other way on the GPU, the
    oracle's assignment is fed to the GPU backward (its idx, gates and logits written into `saved`) and
    the backward runs again, so that both sides differentiate the same routed layer.  Nothing
    flows from the GPU into the oracle."""
    R = L.routing()
    same = check_routing(from_dev(out["idx"]), from_dev(out["gates"]), R, c["k"])
    _, _, lg = buf.saved_views()
    if lg is not None:   # the logits the forward keeps for the backward's softmax (bias included)
        lgv = from_dev(lg).astype(np.float64)
        assert np.max(np.abs(lgv - R.logits) / (1.0 + np.abs(R.logits))) < 2e-5
    else:
        assert c["renorm"]
    y_ref, _ = L.forward()
    g = L.backward()
    rows = np.flatnonzero(same)
    if c["cf"] > 0 and not same.all():
        rows = rows[rows < int(np.flatnonzero(~same)[0])]
    check_close("y", from_dev_bf16(out["y"])[rows], y_ref[rows], float(np.abs(y_ref).max()))
    if not same.all():
        out = backward_on_oracle_assignment(moe, c, inp, R, buf)
    check_close("dx", from_dev_bf16(out["dx"]), g["dx"])
    check_close("dW_r", from_dev(out["dW_r"]), g["dW_r"])
    check_close("db_r", from_dev(out["db_r"]), g["db_r"])
    check_weight_grad("dW_gate", from_dev_bf16(out["dWg"]), g["dW_gate"])
    check_weight_grad("dW_up", from_dev_bf16(out["dWu"]), g["dW_up"])
    check_weight_grad("dW_down", from_dev_bf16(out["dWd"]), g["dW_down"])


def backward_on_oracle_assignment(moe, c, inp, R, buf):
    """The GPU backward from the oracle's idx and gates (gates rounded to fp32).  Without kept
    activations: written into `saved` with the oracle's logits (rounded to fp32; gates not
    renormalised), then moe_layer_bwd.  With them, the backward needs the
    forward's kept a and b of the same dispatch, which moe_layer_fwd (its own routing) cannot give:
    the granular calls run instead on the oracle's assignment -- moe_dispatch, moe_expert_ffn_fwd
    (keeping a, b in the workspace), moe_expert_ffn_bwd, moe_router_bwd, moe_combine_bwd."""
    mc = moe.config_from(c)
    T, d, f, E, S, k = c["T"], c["d"], c["f"], c["E"], c["S"], c["k"]
    G = E + S
    idx = to_dev(R.idx.astype(np.int32))
    gates = to_dev(R.gates.astype(np.float32))
    x, Wg, Wu, Wd, dy = (to_dev_bf16(inp[n]) for n in ("x", "W_gate", "W_up", "W_down", "dy"))
    W_r = to_dev(inp["W_r"])
    b_r = to_dev(inp["b_r"]) if inp["b_r"] is not None else None
    out = dict(dx=torch.empty(T, d, dtype=torch.bfloat16, device="cuda"),
               dW_r=torch.empty(d, E, dtype=torch.float32, device="cuda"),
               db_r=torch.empty(E, dtype=torch.float32, device="cuda"),
               dWg=torch.empty(G, f, d, dtype=torch.bfloat16, device="cuda"),
               dWu=torch.empty(G, f, d, dtype=torch.bfloat16, device="cuda"),
               dWd=torch.empty(G, d, f, dtype=torch.bfloat16, device="cuda"))
    if c.get("keep_rows", 0) > 0:
        scratch = [torch.empty(n, dtype=torch.int32, device="cuda") for n in (E, E + 1, T * k, T * k)]
        x_perm = torch.empty(buf.rows, d, dtype=torch.bfloat16, device="cuda")
        o_perm = torch.empty(buf.rows, d, dtype=torch.bfloat16, device="cuda")
        dx_perm = torch.empty(buf.rows, d, dtype=torch.bfloat16, device="cuda")
        dgates = torch.empty(T, k, dtype=torch.float32, device="cuda")
        dlogits = torch.empty(T, E, dtype=torch.float32, device="cuda")
        moe.moe_dispatch(mc, idx, x, *scratch, x_perm, buf.ws)
        moe.moe_expert_ffn_fwd(mc, x_perm, Wg, Wu, Wd, o_perm, buf.ws)
        moe.moe_expert_ffn_bwd(mc, x_perm, dy, gates, Wg, Wu, Wd, dx_perm, dgates, out["dWg"], out["dWu"],
                               out["dWd"], buf.ws)
        moe.moe_router_bwd(mc, x, W_r, b_r, idx, gates, dgates, dlogits, out["dW_r"], out["db_r"], buf.ws)
        moe.moe_combine_bwd(mc, dx_perm, dlogits, W_r, out["dx"], buf.ws)
    else:
        idx_v, gates_v, logits_v = buf.saved_views()
        idx_v.copy_(idx)
        gates_v.copy_(gates)
        if logits_v is not None:   # the backward's softmax reads the oracle's logits as well
            logits_v.copy_(to_dev(R.logits.astype(np.float32)))
        moe.moe_layer_bwd(mc, x, W_r, b_r, Wg, Wu, Wd, buf.saved, dy, out["dx"], out["dW_r"], out["db_r"],
                          out["dWg"], out["dWu"], out["dWd"], buf.ws)
    status = moe.moe_check_error(buf.ws)
    assert status == 0, moe.moe_status_string(status)
    return out


# The path check_layer takes after a near-tie, run on purpose: the backward from the oracle's
# assignment must match the oracle's gradients (with and without kept activations, with capacity).
@pytest.mark.parametrize("name,keep", [("deepseek_small", 0), ("gptoss_small", 0), ("ragged_mixtral", -1)])
def test_backward_on_oracle_assignment(moe, name, keep):
    c, inp, L = case(name)
    c = dict(c)
    mc = moe.config_from(c)
    c["keep_rows"] = moe.moe_perm_rows(mc) if keep < 0 else keep
    mc = moe.config_from(c)
    buf = moe.Buffers.allocate(mc)
    out = backward_on_oracle_assignment(moe, c, inp, L.routing(), buf)
    g = L.backward()
    check_close("dx", from_dev_bf16(out["dx"]), g["dx"])
    check_close("dW_r", from_dev(out["dW_r"]), g["dW_r"])
    check_weight_grad("dW_gate", from_dev_bf16(out["dWg"]), g["dW_gate"])
    check_weight_grad("dW_up", from_dev_bf16(out["dWu"]), g["dW_up"])
    check_weight_grad("dW_down", from_dev_bf16(out["dWd"]), g["dW_down"])


# The granularity chosen from a byte budget: keep as many rows as the budget holds, and from the
# device's free memory at the time of the call.
@pytest.mark.parametrize("name,tiles", [("ragged_mixtral", 3), ("deepseek_small", 2)])
def test_layer_kept_rows_from_budget(moe, name, tiles):
    c, inp, L = case(name)
    mc = moe.config_from(c)
    budget = tiles * 256 * 4 * c["f"] + 100
    rows, kept = moe.moe_keep_rows_for_budget(mc, budget)
    assert rows == tiles * 256 and kept <= budget
    c = dict(c, keep_rows=rows)
    out, buf = run_layer(moe, c, inp)
    assert buf.saved.numel() >= 8 * c["T"] * c["k"] + kept
    check_layer(moe, c, inp, L, out, buf)


def test_keep_rows_follow_free_memory(moe):
    c, _, _ = case("ragged_mixtral")
    mc = moe.config_from(c)
    cap = moe.moe_perm_rows(mc)
    free, _ = torch.cuda.mem_get_info()
    assert moe.moe_keep_rows_for_free_memory(mc, 0)[0] == cap           # plenty free: keep all
    assert moe.moe_keep_rows_for_free_memory(mc, 1 << 62)[0] == 0       # nothing left: recompute all
    per_tile = 256 * 4 * c["f"]
    rows, _ = moe.moe_keep_rows_for_free_memory(mc, max(0, free - 2 * per_tile - per_tile // 2))
    assert rows in (0, 256, 512)    # about two tiles' bytes free above the reserve


@pytest.mark.parametrize("name", ["tiny", "deepseek_small", "gptoss_small"])
def test_layer_is_deterministic(moe, name):
    c, inp, _ = case(name)
    a, buf = run_layer(moe, c, inp)
    b, _ = run_layer(moe, c, inp, buf)
    for key in a:
        assert torch.equal(a[key].view(torch.uint8), b[key].view(torch.uint8)), key


# Gathered operand loads (gather_in_gemm = 1): the GEMMs gather x and dy from token order instead of
# reading x_perm / dY_perm.  For finite inputs every output equals the default path's bit for bit: a
# pad row reads token 0's row instead of zeros, and its zero gate zeroes every term it feeds.
@pytest.mark.parametrize("name,keep", [(n, 0) for n in CASES] + [("ragged_mixtral", 256), ("deepseek_small", -1),
                                                                 ("gptoss_small", 512)])
def test_gather_in_gemm_bitwise(moe, name, keep):
    c, inp, _ = case(name)
    c = dict(c)
    c["keep_rows"] = moe.moe_perm_rows(moe.config_from(c)) if keep < 0 else keep
    a, buf = run_layer(moe, c, inp)
    b, _ = run_layer(moe, dict(c, gather_in_gemm=1), inp)
    for key in a:
        assert torch.equal(a[key].view(torch.uint8), b[key].view(torch.uint8)), key


@pytest.mark.parametrize("name", ["ragged_mixtral", "deepseek_small", "gptoss_small"])
def test_gather_in_gemm_against_oracle(moe, name):
    c, inp, L = case(name)
    c = dict(c, gather_in_gemm=1)
    out, buf = run_layer(moe, c, inp)
    check_layer(moe, c, inp, L, out, buf)


# The layer backward takes the router's softmax from the logits the forward kept in `saved`: a
# constant added to them changes nothing (softmax is shift-invariant), and equal logits give the
# gradients of a uniform p.  Both runs start from the oracle's assignment written into `saved`.
def test_backward_reads_the_kept_logits(moe):
    import oracle
    c, inp, L = case("ragged_mixtral")
    mc = moe.config_from(c)
    buf = moe.Buffers.allocate(mc)
    T, d, f, E, k = c["T"], c["d"], c["f"], c["E"], c["k"]
    R = L.routing()
    g = L.backward()
    x, Wg, Wu, Wd, dy = (to_dev_bf16(inp[n]) for n in ("x", "W_gate", "W_up", "W_down", "dy"))
    W_r = to_dev(inp["W_r"])
    idx_v, gates_v, logits_v = buf.saved_views()
    gates32 = R.gates.astype(np.float32)

    def backward(logits):
        idx_v.copy_(to_dev(R.idx.astype(np.int32)))
        gates_v.copy_(to_dev(gates32))
        logits_v.copy_(to_dev(logits.astype(np.float32)))
        out = [torch.empty(d, E, dtype=torch.float32, device="cuda"), torch.empty(T, d, dtype=torch.bfloat16,
                                                                                  device="cuda")]
        dW = [torch.empty(E, f, d, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        dWd = torch.empty(E, d, f, dtype=torch.bfloat16, device="cuda")
        moe.moe_layer_bwd(mc, x, W_r, None, Wg, Wu, Wd, buf.saved, dy, out[1], out[0], None, dW[0], dW[1], dWd,
                          buf.ws)
        assert moe.moe_check_error(buf.ws) == 0
        return from_dev(out[0]).astype(np.float64)

    dw_kept = backward(R.logits)
    check_close("dW_r", dw_kept, g["dW_r"])
    dw_shift = backward(R.logits + 5.0)
    assert np.max(np.abs(dw_shift - dw_kept)) <= 1e-3 * np.max(np.abs(dw_kept))
    dw_flat = backward(np.zeros((T, E)))
    dl = oracle.router_backward_logits(np.full((T, E), 1.0 / E), R.idx, gates32.astype(np.float64), g["dgates"],
                                       False)
    ref = oracle.bf16_to_f64(inp["x"]).T @ dl
    check_close("dW_r (uniform p)", dw_flat, ref)
    assert np.max(np.abs(dw_flat - dw_kept)) > 0.1 * np.max(np.abs(dw_kept))
