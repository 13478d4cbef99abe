"""Parity at the five workloads' full sizes (GPU).

The fused moe_layer_fwd / moe_layer_bwd run exactly as bench.py times them.  The fp64 oracle
checks, one by one, what it can afford at these sizes:
  * routing of every token (bit-exact top-k where decided, gates to 1e-5 relative);
  * counts, offsets and the permutation of every slot (moe_dispatch on the oracle's assignments);
  * y, dx and dgates of a seeded sample of tokens (their experts' forward and backward in fp64);
  * full rows/columns of dW_gate, dW_up and dW_down for sampled (expert, hidden unit) pairs, each
    an exact reduction over all the rows that expert received (the backward runs on the oracle's
    assignment when a near-tie routed a token differently in the forward);
  * the router backward on all tokens, with seeded gate gradients as its input.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import (check_close, check_routing, decided_tokens, from_dev, from_dev_bf16, segment_rows,
                     to_dev, to_dev_bf16)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

WORKLOADS = ["mixtral", "deepseek", "qwen3", "gptoss"]
N_TOKENS = 24
N_UNITS = 2


@pytest.fixture(scope="module", params=WORKLOADS)
def full(request, moe):
    name = request.param
    cfg = synth.CONFIGS[name]
    inp = synth.make_inputs(cfg, seed=0)
    L = oracle.Layer(inp, cfg)
    T, d, f, E, k, S = cfg["T"], cfg["d"], cfg["f"], cfg["E"], cfg["k"], cfg["S"]
    G = E + S
    mc = moe.config_from(cfg)
    buf = moe.Buffers.allocate(mc)
    dev = dict(x=to_dev_bf16(inp["x"]), W_r=to_dev(inp["W_r"]),
               b_r=to_dev(inp["b_r"]) if inp["b_r"] is not None else None,
               Wg=to_dev_bf16(inp["W_gate"]), Wu=to_dev_bf16(inp["W_up"]), Wd=to_dev_bf16(inp["W_down"]),
               dy=to_dev_bf16(inp["dy"]))
    y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    dx = torch.empty_like(y)
    dW_r = torch.empty(d, E, dtype=torch.float32, device="cuda")
    db_r = torch.empty(E, dtype=torch.float32, device="cuda")
    dWg, dWu = torch.empty_like(dev["Wg"]), torch.empty_like(dev["Wu"])
    dWd = torch.empty_like(dev["Wd"])
    moe.moe_layer_fwd(mc, dev["x"], dev["W_r"], dev["b_r"], dev["Wg"], dev["Wu"], dev["Wd"], y, buf.saved, buf.ws)
    idx_fwd = from_dev(buf.saved.view(torch.int32)[:T * k].view(T, k))
    gates_fwd = from_dev(buf.saved.view(torch.float32)[T * k:2 * T * k].view(T, k))
    # The gradients depend on every token's assignment.  Where a near-tie went the other way on the
    # GPU, the backward runs from the oracle's assignment (idx, fp32 gates and logits in `saved`),
    # so the gradient checks below compare the same routed layer; nothing flows into the oracle.
    R = L.routing()
    if not np.array_equal(idx_fwd, R.idx):
        idx_v, gates_v, logits_v = buf.saved_views()
        idx_v.copy_(to_dev(R.idx.astype(np.int32)))
        gates_v.copy_(to_dev(R.gates.astype(np.float32)))
        if logits_v is not None:
            logits_v.copy_(to_dev(R.logits.astype(np.float32)))
    moe.moe_layer_bwd(mc, dev["x"], dev["W_r"], dev["b_r"], dev["Wg"], dev["Wu"], dev["Wd"], buf.saved, dev["dy"],
                      dx, dW_r, db_r, dWg, dWu, dWd, buf.ws)
    assert moe.moe_check_error(buf.ws) == 0
    out = dict(y=y, dx=dx, dW_r=dW_r, db_r=db_r, dWg=dWg, dWu=dWu, dWd=dWd, idx=idx_fwd, gates=gates_fwd)
    yield name, cfg, inp, L, mc, buf, dev, out
    del dev, out, buf
    torch.cuda.empty_cache()


def test_routing_every_token(full):
    name, cfg, inp, L, mc, buf, dev, out = full
    same = check_routing(out["idx"], out["gates"], L.routing(), cfg["k"])
    assert same.mean() > 0.995


def test_dispatch_every_slot(full, moe):
    name, cfg, inp, L, mc, buf, dev, out = full
    T, k, E, d = cfg["T"], cfg["k"], cfg["E"], cfg["d"]
    D = L.dispatch()
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    ros = torch.empty(T * k, dtype=torch.int32, device="cuda")
    tor = torch.empty(T * k, dtype=torch.int32, device="cuda")
    x_perm = torch.empty(buf.rows, d, dtype=torch.bfloat16, device="cuda")
    ws2 = moe.Buffers.allocate(mc)
    moe.moe_dispatch(mc, to_dev(L.routing().idx.astype(np.int32)), dev["x"], counts, offsets, ros, tor,
                     x_perm, ws2.ws)
    assert moe.moe_check_error(ws2.ws) == 0
    assert np.array_equal(from_dev(counts), D.counts)
    assert np.array_equal(from_dev(offsets), D.offsets)
    assert np.array_equal(from_dev(ros).reshape(T, k), D.row_of_slot)
    assert np.array_equal(from_dev(tor)[:D.offsets[-1]], D.token_of_row)
    if cfg["cf"] > 0:
        assert D.kept.max() <= oracle.capacity_of(T, k, E, cfg["cf"])
    # gathered rows: a seeded sample of kept slots (exact copies) and every pad row (zeros)
    kept, P = segment_rows(D, T, cfg["S"])
    rng = np.random.default_rng(7)
    ts, js = np.nonzero(D.row_of_slot >= 0)
    pick = rng.choice(ts.size, size=min(4096, ts.size), replace=False)
    rows = np.array([P[L.routing().idx[t, j]] + D.position[t, j] for t, j in zip(ts[pick], js[pick])])
    got = from_dev_bf16(x_perm[torch.from_numpy(rows).cuda()])
    assert np.array_equal(got, L.x[ts[pick]]), "gathered rows differ from x"
    pads = np.concatenate([np.arange(P[g] + kept[g], P[g + 1]) for g in range(len(kept))]).astype(np.int64)
    if pads.size:
        assert torch.count_nonzero(x_perm[torch.from_numpy(pads).cuda()]).item() == 0, "pad rows not zero"


def _sample_tokens(cfg, L, out, seed):
    """Tokens whose slots the oracle and the GPU assign alike.  With a capacity, a slot's queue
    position (hence whether it is dropped) depends on the routing of every earlier token, so when
    the two routings part at a near-tie the sample is drawn from the tokens before the first such
    token, whose queue positions agree by construction."""
    order_ok, _ = decided_tokens(L.routing().logits, cfg["k"])
    same = np.all(out["idx"] == L.routing().idx, axis=1)
    agree = same & order_ok
    if cfg["cf"] > 0 and not same.all():
        agree[int(np.flatnonzero(~same)[0]):] = False
    rng = np.random.default_rng(seed)
    pool = np.flatnonzero(agree)
    assert pool.size >= N_TOKENS, "too few tokens before the first routing difference"
    return np.sort(rng.choice(pool, size=N_TOKENS, replace=False))


def test_sampled_tokens(full):
    """y and dx of sampled tokens whose forward routing agrees (the backward ran on the oracle's
    assignment if any token's did not)."""
    name, cfg, inp, L, mc, buf, dev, out = full
    toks = _sample_tokens(cfg, L, out, seed=3)
    s = L.token_outputs(toks)
    t_dev = torch.from_numpy(toks).cuda()
    check_close("y[sample]", from_dev_bf16(out["y"][t_dev]), s["y"])
    check_close("dx[sample]", from_dev_bf16(out["dx"][t_dev]), s["dx"])


def test_sampled_weight_gradients(full):
    name, cfg, inp, L, mc, buf, dev, out = full
    E, S, f = cfg["E"], cfg["S"], cfg["f"]
    rng = np.random.default_rng(5)
    kept = L.dispatch().kept
    experts = list(rng.choice(np.flatnonzero(kept > 0), size=min(3, int((kept > 0).sum())), replace=False))
    experts += [E + s for s in range(S)]
    for e in experts:
        cols = np.sort(rng.choice(f, size=N_UNITS, replace=False))
        ref = L.weight_grad_columns(int(e), cols)
        c_dev = torch.from_numpy(cols).cuda()
        got_g = from_dev_bf16(out["dWg"][int(e)][c_dev])
        got_u = from_dev_bf16(out["dWu"][int(e)][c_dev])
        got_d = from_dev_bf16(out["dWd"][int(e)][:, c_dev])
        check_close(f"dW_gate[{e}][cols]", got_g, ref["dW_gate"])
        check_close(f"dW_up[{e}][cols]", got_u, ref["dW_up"])
        check_close(f"dW_down[{e}][:, cols]", got_d, ref["dW_down"])


def test_router_backward_all_tokens(full, moe):
    name, cfg, inp, L, mc, buf, dev, out = full
    T, k, E, d = cfg["T"], cfg["k"], cfg["E"], cfg["d"]
    R = L.routing()
    gates32 = R.gates.astype(np.float32)
    dg32 = synth.normal_f32(13, "aux", (T, k), 1.0, chunk=9)
    dl_ref = oracle.router_backward_logits(R.p, R.idx, gates32.astype(np.float64), dg32.astype(np.float64),
                                           bool(cfg["renorm"]))
    dWr_ref, db_ref, _ = oracle.router_backward(L.x, inp["W_r"], dl_ref)
    dlogits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    dW_r = torch.empty(d, E, dtype=torch.float32, device="cuda")
    db_r = torch.empty(E, dtype=torch.float32, device="cuda")
    moe.moe_router_bwd(mc, dev["x"], dev["W_r"], dev["b_r"], to_dev(R.idx.astype(np.int32)), to_dev(gates32),
                       to_dev(dg32), dlogits, dW_r, db_r, buf.ws)
    assert moe.moe_check_error(buf.ws) == 0
    check_close("dlogits", from_dev(dlogits), dl_ref)
    check_close("dW_r", from_dev(dW_r), dWr_ref)
    check_close("db_r", from_dev(db_r), db_ref)


@pytest.mark.parametrize("name", WORKLOADS)
def test_gather_in_gemm_bitwise_full_size(moe, name):
    """Gathered operand loads at full size, in the bench's launch configuration: every output of
    moe_layer_fwd / moe_layer_bwd equals the default path's bit for bit (finite inputs)."""
    cfg = synth.CONFIGS[name]
    inp = synth.make_inputs(cfg, seed=0)
    T, d, f, E, S = cfg["T"], cfg["d"], cfg["f"], cfg["E"], cfg["S"]
    G = E + S
    dev = dict(x=to_dev_bf16(inp["x"]), W_r=to_dev(inp["W_r"]),
               b_r=to_dev(inp["b_r"]) if inp["b_r"] is not None else None,
               Wg=to_dev_bf16(inp["W_gate"]), Wu=to_dev_bf16(inp["W_up"]), Wd=to_dev_bf16(inp["W_down"]),
               dy=to_dev_bf16(inp["dy"]))
    res = []
    for gig in (0, 1):
        mc = moe.config_from(dict(cfg, gather_in_gemm=gig))
        buf = moe.Buffers.allocate(mc)
        out = dict(y=torch.empty(T, d, dtype=torch.bfloat16, device="cuda"),
                   dx=torch.empty(T, d, dtype=torch.bfloat16, device="cuda"),
                   dW_r=torch.empty(d, E, dtype=torch.float32, device="cuda"),
                   db_r=torch.empty(E, dtype=torch.float32, device="cuda"),
                   dWg=torch.empty(G, f, d, dtype=torch.bfloat16, device="cuda"),
                   dWu=torch.empty(G, f, d, dtype=torch.bfloat16, device="cuda"),
                   dWd=torch.empty(G, d, f, dtype=torch.bfloat16, device="cuda"))
        moe.moe_layer_fwd(mc, dev["x"], dev["W_r"], dev["b_r"], dev["Wg"], dev["Wu"], dev["Wd"], out["y"], buf.saved,
                          buf.ws)
        moe.moe_layer_bwd(mc, dev["x"], dev["W_r"], dev["b_r"], dev["Wg"], dev["Wu"], dev["Wd"], buf.saved, dev["dy"],
                          out["dx"], out["dW_r"], out["db_r"], out["dWg"], out["dWu"], out["dWd"], buf.ws)
        assert moe.moe_check_error(buf.ws) == 0
        out["saved"] = buf.saved
        res.append(out)
        del buf
    for key in res[0]:
        assert torch.equal(res[0][key].view(torch.uint8), res[1][key].view(torch.uint8)), key
    del res, dev
    torch.cuda.empty_cache()


def test_empty_experts_have_zero_weight_gradients(full):
    """Experts that received no rows have exactly zero weight gradients: the epilogue stores their
    tiles beside the MMA tiles of the other experts (the Qwen3-like routing leaves about half the
    experts empty); every other expert's gradient is checked on sampled hidden units above."""
    name, cfg, inp, L, mc, buf, dev, out = full
    kept = L.dispatch().kept
    empty = np.flatnonzero(kept == 0)
    if name == "qwen3":
        assert empty.size > 32
    for e in empty:
        for key in ("dWg", "dWu", "dWd"):
            assert torch.count_nonzero(out[key][int(e)]).item() == 0, (key, int(e))
