"""The FP8 (e4m3) backward on the GPU against the oracle's quantised backward (GPU).

* the column quantiser (W_down's columns; column i of W_gate and W_up together): codes and scales
  bit-exact, both sides deciding in fp32;
* moe_layer_bwd_fp8 on the small workloads: dx, dW_r, db_r and the expert weight gradients against
  oracle.fp8.layer_backward_fp8 under the bf16 output rule, given identical assignments (the
  oracle's idx, gates and logits are written into `saved`, so the backward differentiates the oracle's
  routed layer; nothing flows from the GPU into the oracle);
* the same at the four large workloads' full sizes on sampled tokens (dx, dgates) and sampled
  hidden units (whole weight-gradient rows and columns).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import fp8
from cases import case
from harness import check_close, check_weight_grad, from_dev, from_dev_bf16, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _bits(v):
    return synth.f32_to_bf16_bits(np.asarray(v, np.float32))


@pytest.mark.parametrize("G,r1,r2,cols", [(3, 64, 0, 64), (2, 2880, 0, 96), (3, 128, 128, 200), (1, 48, 16, 33),
                                          (2, 16384, 16384, 64)])
def test_quantize_cols_bit_exact(moe, G, r1, r2, cols):
    rng = np.random.default_rng(G * 1000 + r1 + cols)
    top = rng.normal(0, 1, (G, r1, cols)) * np.exp(rng.uniform(-12, 12, (G, 1, cols)))
    bot = rng.normal(0, 1, (G, r2, cols)) * np.exp(rng.uniform(-12, 12, (G, 1, cols)))
    top[:, :, 3 % cols] = 0.0                                  # an all-zero column (with r2 = 0)
    top[0, ::5, 1] = -0.0                                      # signed zeros
    top[0, :, 2 % cols] *= 1e-30 / np.abs(top[0, :, 2 % cols]).max()   # scale below 2^-80
    if cols > 4:
        # quotients exactly on e4m3 rounding ties (column maximum 448 * 2^-5 => scale 2^-5)
        ties = np.array([1.0625, 1.1875, -1.0625, 2.0 ** -10, 3 * 2.0 ** -10, 17.0, 19.0, 400.0])
        top[:, :, 4] = np.resize(ties, r1)[None, :] * 2.0 ** -5
        top[:, 0, 4] = 448.0 * 2.0 ** -5
        if r2:
            bot[:, :, 4] = 0.5 * 2.0 ** -5
    tb, bb = _bits(top), _bits(bot)
    rows = r1 + r2
    codes = torch.empty(G, cols, rows, dtype=torch.uint8, device="cuda")
    scales = torch.empty(G, cols, dtype=torch.float32, device="cuda")
    moe.moe_quantize_cols_e4m3(to_dev_bf16(tb), to_dev_bf16(bb) if r2 else None, codes, scales)
    torch.cuda.synchronize()
    for g in range(G):
        src = oracle.bf16_to_f64(np.concatenate([tb[g], bb[g]], axis=0) if r2 else tb[g]).astype(np.float32)
        q, s = fp8.quantize_cols_e4m3(src)
        assert np.array_equal(from_dev(scales)[g], s), g
        assert np.array_equal(from_dev(codes)[g], q), g


def _weight_codes(moe, Wg, Wu, Wd, G, f, d):
    """The forward's row codes of W_gate and W_up, and the backward's column codes of W_down and of
    W_gate over W_up, from the GPU quantisers (bit-exact with the oracle's)."""
    def rows(W):
        c = torch.empty(W.shape, dtype=torch.uint8, device="cuda")
        s = torch.empty(W.shape[0], W.shape[1], dtype=torch.float32, device="cuda")
        moe.moe_quantize_rows_e4m3(W, c, s)
        return c, s
    wdt = torch.empty(G, f, d, dtype=torch.uint8, device="cuda")
    wdts = torch.empty(G, f, dtype=torch.float32, device="cuda")
    moe.moe_quantize_cols_e4m3(Wd, None, wdt, wdts)
    wgut = torch.empty(G, d, 2 * f, dtype=torch.uint8, device="cuda")
    wguts = torch.empty(G, d, dtype=torch.float32, device="cuda")
    moe.moe_quantize_cols_e4m3(Wg, Wu, wgut, wguts)
    return (*rows(Wg), *rows(Wu), wdt, wdts, wgut, wguts)


def run_bwd_fp8(moe, c, inp, R):
    """moe_layer_bwd_fp8 from the oracle's assignment R (idx; gates and logits rounded to fp32) in
    `saved`."""
    mc = moe.config_from(c)
    buf = moe.Buffers.allocate(mc)
    T, d, f, E, S, k = c["T"], c["d"], c["f"], c["E"], c["S"], c["k"]
    G = E + S
    idx_v, gates_v, logits_v = buf.saved_views()
    idx_v.copy_(to_dev(R.idx.astype(np.int32)))
    gates_v.copy_(to_dev(R.gates.astype(np.float32)))
    if logits_v is not None:
        logits_v.copy_(to_dev(R.logits.astype(np.float32)))
    x, Wg, Wu, Wd, dy = (to_dev_bf16(inp[n]) for n in ("x", "W_gate", "W_up", "W_down", "dy"))
    codes = _weight_codes(moe, Wg, Wu, Wd, G, f, d)
    out = dict(dx=torch.full((T, d), float("nan"), dtype=torch.bfloat16, device="cuda"),
               dW_r=torch.empty(d, E, dtype=torch.float32, device="cuda"),
               db_r=torch.empty(E, dtype=torch.float32, device="cuda"),
               dWg=torch.full((G, f, d), float("nan"), dtype=torch.bfloat16, device="cuda"),
               dWu=torch.full((G, f, d), float("nan"), dtype=torch.bfloat16, device="cuda"),
               dWd=torch.full((G, d, f), float("nan"), dtype=torch.bfloat16, device="cuda"))
    b_r = to_dev(inp["b_r"]) if inp["b_r"] is not None else None
    moe.moe_layer_bwd_fp8(mc, x, to_dev(inp["W_r"]), b_r, *codes, buf.saved, dy, out["dx"], out["dW_r"],
                          out["db_r"], out["dWg"], out["dWu"], out["dWd"], buf.ws)
    status = moe.moe_check_error(buf.ws)
    assert status == 0, moe.moe_status_string(status)
    return out


@pytest.mark.parametrize("name", ["tiny", "ragged_mixtral", "deepseek_small", "qwen_small", "gptoss_small",
                                  "single_expert", "k_equals_E", "max_shared", "router_e96_k8", "router_e64_renorm",
                                  "router_simt_e160", "max_d_model", "max_d_ff"])
def test_layer_bwd_fp8(moe, name):
    c, inp, L = case(name)
    out = run_bwd_fp8(moe, c, inp, L.routing())
    g = fp8.layer_backward_fp8(L)
    check_close("dx (fp8 backward)", from_dev_bf16(out["dx"]), g["dx"])
    check_close("dW_r (fp8 backward)", from_dev(out["dW_r"]), g["dW_r"])
    check_close("db_r (fp8 backward)", from_dev(out["db_r"]), g["db_r"])
    check_weight_grad("dW_gate (fp8 backward)", from_dev_bf16(out["dWg"]), g["dW_gate"])
    check_weight_grad("dW_up (fp8 backward)", from_dev_bf16(out["dWu"]), g["dW_up"])
    check_weight_grad("dW_down (fp8 backward)", from_dev_bf16(out["dWd"]), g["dW_down"])


def test_layer_bwd_fp8_rejects_kept_activations(moe):
    c, inp, L = case("tiny")
    mc = moe.config_from(dict(c, keep_rows=256))
    buf = moe.Buffers.allocate(mc)
    t = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoEError) as e:
        moe.moe_layer_bwd_fp8(mc, *([t] * 19), buf.ws)
    assert e.value.code == 1


@pytest.mark.slow
@pytest.mark.parametrize("name,n_tok", [("mixtral", 6), ("deepseek", 4), ("qwen3", 4), ("gptoss", 4)])
def test_layer_bwd_fp8_full_size(moe, name, n_tok):
    """The FP8 backward at the workload's full size, on the oracle's assignment: dx and dgates of
    sampled tokens, and whole weight-gradient rows/columns of sampled hidden units, one by one.  The
    oracle quantises only the experts the sampled tokens visit, so the Mixtral-like sample is drawn
    from the tokens of the most common expert pair."""
    cfg = synth.CONFIGS[name]
    inp = synth.make_inputs(cfg, seed=0)
    L = oracle.Layer(inp, cfg)
    R = L.routing()
    out = run_bwd_fp8(moe, cfg, inp, R)
    rng = np.random.default_rng(21)
    pool = np.arange(cfg["T"])
    if name == "mixtral":
        pairs = np.sort(R.idx, axis=1)
        key = pairs[:, 0] * cfg["E"] + pairs[:, 1]
        pool = pool[key == np.bincount(key).argmax()]
    toks = np.sort(rng.choice(pool, size=n_tok, replace=False))
    s = fp8.token_grads_fp8(L, toks)
    check_close("dx[sample] (fp8 backward)", from_dev_bf16(out["dx"][torch.from_numpy(toks).cuda()]), s["dx"])
    kept = L.dispatch().kept
    experts = list(rng.choice(np.flatnonzero(kept > 0), size=min(2, int((kept > 0).sum())), replace=False))
    experts += [cfg["E"] + j for j in range(cfg["S"])]
    for e in experts:
        cols = np.sort(rng.choice(cfg["f"], size=2, replace=False))
        ref = fp8.weight_grad_columns_fp8(L, int(e), cols)
        c_dev = torch.from_numpy(cols).cuda()
        check_close(f"dW_gate[{e}][cols] (fp8)", from_dev_bf16(out["dWg"][int(e)][c_dev]), ref["dW_gate"])
        check_close(f"dW_up[{e}][cols] (fp8)", from_dev_bf16(out["dWu"][int(e)][c_dev]), ref["dW_up"])
        check_close(f"dW_down[{e}][:, cols] (fp8)", from_dev_bf16(out["dWd"][int(e)][:, c_dev]), ref["dW_down"])
