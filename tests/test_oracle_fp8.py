"""Pins of the oracle's FP8 (e4m3) quantisation step (CPU)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
import synth


def test_decode_landmarks():
    v = fp8.e4m3_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x39, 0x7E, 0xFE, 0x80], np.uint8))
    assert list(v) == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.125, 448.0, -448.0, 0.0]
    assert np.isnan(fp8.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    assert np.array_equal(fp8.e4m3_encode_rne(fp8.e4m3_decode(codes)), codes)


def test_ties_go_to_even_and_large_values_saturate():
    v = np.array([1.0625, 1.1875, 2.0 ** -9 * 0.5, 2.0 ** -9 * 1.5, 464.0, 1000.0, -1000.0])
    got = fp8.e4m3_decode(fp8.e4m3_encode_rne(v))
    assert list(got) == [1.0, 1.25, 0.0, 2.0 * 2.0 ** -9, 448.0, 448.0, -448.0]


def test_matches_torch_float8_conversion():
    # an independent implementation of the same rounding (round to nearest even, in range)
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1e-2, 20000),
                        rng.normal(0, 1, 20000)]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode_rne(v), ref)


def test_row_scaling_uses_the_whole_range():
    rng = np.random.default_rng(1)
    rows = rng.normal(0, 3, (64, 200)).astype(np.float32)
    q, s = fp8.quantize_rows_e4m3(rows)
    dec = fp8.e4m3_decode(q)
    assert np.all(np.abs(dec).max(axis=1) == 448.0)
    # relative error of every element within half an e4m3 step of its binade (2^-4), plus the
    # subnormal floor
    err = np.abs(dec * s[:, None] - rows)
    assert np.all(err <= np.abs(rows) * 2.0 ** -4 + s[:, None] * 2.0 ** -10)
    z, zs = fp8.quantize_rows_e4m3(np.zeros((2, 8), np.float32))
    assert not z.any() and np.all(zs == 1.0)


def test_lossless_inputs_reduce_to_the_bf16_expert():
    # values already on the e4m3 grid, with row maxima 448 * 2^j: quantisation is exact, so the
    # quantised projection equals the plain expert forward's h on the same values
    rng = np.random.default_rng(2)
    grid = fp8.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    grid = grid[grid >= 2.0 ** -3]

    def rows(n, w, j):
        r = rng.choice(grid, (n, w)) * rng.choice([-1.0, 1.0], (n, w))
        r[:, 0] = 448.0
        return (r * 2.0 ** j).astype(np.float32)
    x, wg, wu = rows(5, 64, -6), rows(32, 64, -9), rows(32, 64, -9)
    xq, xs = fp8.quantize_rows_e4m3(x)
    gq, gs = fp8.quantize_rows_e4m3(wg)
    uq, us = fp8.quantize_rows_e4m3(wu)
    h = fp8.gate_up_fp8(xq, xs, gq, gs, uq, us)
    _, _, h_ref, _ = oracle.expert_forward(x.astype(np.float64), wg.astype(np.float64),
                                           wu.astype(np.float64), np.zeros((1, 32)))
    assert np.allclose(h, h_ref, rtol=1e-12, atol=0)


def _grid_rows(rng, n, w, exps):
    """[n, w] values on the e4m3 grid times 2^exps[i], row i's maximum magnitude 448 * 2^exps[i]:
    the row quantisation of such rows is exact (scale 2^exps[i])."""
    grid = fp8.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    grid = grid[grid >= 2.0 ** -3]
    r = rng.choice(grid, (n, w)) * rng.choice([-1.0, 1.0], (n, w))
    r[np.arange(n), rng.integers(0, w, n)] = 448.0
    return r * np.ldexp(1.0, np.asarray(exps))[:, None]


def test_down_lossless_with_per_channel_scales():
    # rows of W_down with scales 2^-12 .. 2^4 apart: exact only when each output channel gets its
    # own row's scale
    rng = np.random.default_rng(3)
    h = _grid_rows(rng, 7, 64, rng.integers(-4, 4, 7))
    wd = _grid_rows(rng, 48, 64, rng.integers(-12, 5, 48))
    hq, hs = fp8.quantize_rows_e4m3(h.astype(np.float32))
    dq, ds = fp8.quantize_rows_e4m3(wd.astype(np.float32))
    assert np.array_equal(fp8.down_fp8(hq, hs, dq, ds), h @ wd.T)


def _lossless_layer(T=24, d=64, f=64, E=4, k=2, S=1, cf=0.0, renorm=False, seed=5):
    """Layer inputs on which every step of the e4m3 forward is exact.

    x_t = 2^j_t e_0 + 448 2^j_t e_1 (row scale 2^j_t); W_gate[g][i] has 2^a_i at column 0, 0 at
    column 1 and its row maximum 448 2^(a_i - 4) elsewhere; W_up[g][i] has its maximum 448 2^b_i
    at column 0 and 0 at column 1.  So a_ti = 2^(j_t + a_i) >= 64, where silu(a) = a exactly in
    fp64 (and fp32), b_ti = 448 2^(j_t + b_i), and h_ti = 448 2^(2 j_t + a_i + b_i): on the bf16
    grid and, per row, on the e4m3 grid times a power of two.  W_down rows are grid rows."""
    rng = np.random.default_rng(seed)
    G = E + S
    j = rng.integers(0, 4, T)
    x = np.zeros((T, d))
    x[:, 0] = np.ldexp(1.0, j)
    x[:, 1] = 448.0 * np.ldexp(1.0, j)
    Wg = np.empty((G, f, d))
    Wu = np.empty((G, f, d))
    Wd = np.empty((G, d, f))
    for g in range(G):
        a = rng.integers(6, 11, f)
        b = rng.integers(-3, 4, f)
        Wg[g] = _grid_rows(rng, f, d, a - 4) / 2.0   # maxima 224 2^(a-4): below the column-2 entry
        Wg[g][:, 2] = 448.0 * np.ldexp(1.0, a - 4)
        Wg[g][:, 0] = np.ldexp(1.0, a)
        Wg[g][:, 1] = 0.0
        Wu[g] = _grid_rows(rng, f, d, b) / 2.0
        Wu[g][:, 0] = 448.0 * np.ldexp(1.0, b)
        Wu[g][:, 1] = 0.0
        Wd[g] = _grid_rows(rng, d, f, rng.integers(-8, -2, d))
    bits = lambda v: synth.f32_to_bf16_bits(v.astype(np.float32))
    for v in (x, Wg, Wu, Wd):   # every value is exact in bf16
        assert np.array_equal(oracle.bf16_to_f64(bits(v)), v)
    # router logits of a few units (x has entries up to 448 * 8): no saturated gates
    inp = {"x": bits(x), "W_r": rng.normal(0, 1e-3, (d, E)).astype(np.float32), "b_r": None,
           "W_gate": bits(Wg), "W_up": bits(Wu), "W_down": bits(Wd), "dy": bits(np.zeros((T, d)))}
    cfg = {"T": T, "d": d, "E": E, "k": k, "f": f, "S": S, "renorm": renorm, "cf": cf}
    return oracle.Layer(inp, cfg)


@pytest.mark.parametrize("variant", [dict(), dict(S=0, renorm=True, k=3), dict(cf=0.6, S=2)])
def test_lossless_layer_forward_equals_the_exact_layer(variant):
    L = _lossless_layer(**variant)
    y_ref, _ = L.forward()
    y = fp8.layer_forward_fp8(L)
    assert np.abs(y_ref).max() > 0
    assert np.allclose(y, y_ref, rtol=1e-12, atol=0)


def test_quantised_layer_forward_error_is_the_e4m3_size():
    # on ordinary inputs the e4m3 forward is close to, but not the same as, the exact forward:
    # relative error around the e4m3 step (2^-4 per element, averaging out over the sums)
    import cases
    c, inp, L = cases.case("tiny")
    y_ref, _ = L.forward()
    y = fp8.layer_forward_fp8(L)
    rel = np.linalg.norm(y - y_ref) / np.linalg.norm(y_ref)
    assert 1e-3 < rel < 0.1


def test_token_outputs_fp8_equal_the_layer_forward():
    # the one-token-at-a-time form (sampled output channels) against the whole-layer form
    import cases
    for name in ("tiny", "gptoss_small", "deepseek_small"):
        c, inp, L = cases.case(name)
        y = fp8.layer_forward_fp8(L)
        toks = np.array([0, 3, 17, c["T"] - 1])
        cols = np.array([1, 5, c["d"] - 1])
        np.testing.assert_allclose(fp8.token_outputs_fp8(L, toks, cols), y[toks][:, cols], rtol=1e-12, atol=1e-300)


# ---- the e4m3 backward

def test_column_quantisation_scales_are_column_maxima():
    rng = np.random.default_rng(11)
    W = (rng.normal(0, 1, (40, 24)) * np.exp2(rng.integers(-6, 6, 24))[None, :]).astype(np.float32)
    q, s = fp8.quantize_cols_e4m3(W)
    assert q.shape == (24, 40) and s.shape == (24,)
    np.testing.assert_array_equal(s, (np.abs(W).max(axis=0) / np.float32(448.0)).astype(np.float32))
    assert np.all(np.abs(fp8.e4m3_decode(q)).max(axis=1) == 448.0)


def test_data_gradient_products_lossless():
    # rows of the left operands and columns of the weights on the e4m3 grid (maxima 448 * 2^j):
    # every quantisation is exact, so the e4m3 products equal the plain ones
    rng = np.random.default_rng(12)
    n, d, f = 6, 64, 48
    dy = _grid_rows(rng, n, d, rng.integers(-5, 3, n))
    WdT = _grid_rows(rng, f, d, rng.integers(-9, -3, f))        # the columns of W_d
    dyq, dys = fp8.quantize_rows_e4m3(dy.astype(np.float32))
    wq, ws = fp8.quantize_cols_e4m3(WdT.T.astype(np.float32))
    assert np.array_equal(fp8.dh_fp8(dyq, dys, wq, ws), dy @ WdT.T)
    dab = _grid_rows(rng, n, 2 * f, rng.integers(-7, 0, n))
    WguT = _grid_rows(rng, d, 2 * f, rng.integers(-10, -4, d))  # column i of W_g, then of W_u
    aq, as_ = fp8.quantize_rows_e4m3(dab.astype(np.float32))
    wq, ws = fp8.quantize_cols_e4m3(WguT.T.astype(np.float32))
    Wg, Wu = WguT[:, :f].T, WguT[:, f:].T
    assert np.allclose(fp8.dx_fp8(aq, as_, wq, ws), dab[:, :f] @ Wg + dab[:, f:] @ Wu, rtol=1e-13, atol=0)


@pytest.mark.parametrize("name", ["tiny", "deepseek_small", "gptoss_small"])
def test_quantised_backward_error_is_the_e4m3_size(name):
    # every gradient of the e4m3 backward sits within e4m3-sized relative error of the exact one
    import cases
    c, inp, L = cases.case(name)
    g = L.backward()
    q = fp8.layer_backward_fp8(L)
    for key in ("dx", "dW_gate", "dW_up", "dW_down", "dgates", "dW_r"):
        rel = np.linalg.norm(q[key] - g[key]) / np.linalg.norm(g[key])
        assert 1e-4 < rel < 0.1, (key, rel)


def test_backward_weight_scales_are_per_channel():
    # channels spread over 2^-20 .. 1, wider than e4m3's range (~2^18): only one scale per channel
    # keeps every channel's gradient within the e4m3 error; one scale for the whole matrix flushes
    # the small channels to zero
    rng = np.random.default_rng(13)
    n, d, f = 32, 64, 64
    x = rng.normal(0, 1, (n, d))
    dy = rng.normal(0, 1, (n, d))
    g = rng.uniform(0.2, 1.0, n)
    Wg = rng.normal(0, 0.1, (f, d))
    Wu = rng.normal(0, 0.1, (f, d))
    Wd = rng.normal(0, 0.1, (d, f)) * np.exp2(-rng.uniform(0, 20, f))[None, :]   # W_d's columns
    ref = oracle.expert_backward(x, dy, g, Wg, Wu, Wd)
    got = fp8.expert_backward_fp8(x.astype(np.float32), dy.astype(np.float32), g, Wg, Wu, Wd)
    for k, name in ((1, "dW_gate"), (2, "dW_up")):       # rows: the d_ff channels dh' feeds
        err = np.linalg.norm(got[k] - ref[k], axis=1) / np.linalg.norm(ref[k], axis=1)
        assert err.max() < 0.2, (name, err.max())
    sc = np.exp2(-rng.uniform(0, 20, d))[None, :]            # W_g's and W_u's columns
    Wg2, Wu2 = Wg * sc, Wu * sc
    ref = oracle.expert_backward(x, dy, g, Wg2, Wu2, Wd)
    got = fp8.expert_backward_fp8(x.astype(np.float32), dy.astype(np.float32), g, Wg2, Wu2, Wd)
    err = np.linalg.norm(got[0] - ref[0], axis=0) / np.linalg.norm(ref[0], axis=0)   # dx columns
    assert err.max() < 0.2, ("dx", err.max())


def test_sampled_backward_forms_equal_the_layer_backward():
    # token by token (dx, dgates) and hidden unit by unit (weight-gradient rows and columns)
    # against the whole-layer e4m3 backward: capacity drops, shared experts, renormalised gates
    import cases
    for name in ("tiny", "gptoss_small", "deepseek_small"):
        c, inp, L = cases.case(name)
        full = fp8.layer_backward_fp8(L)
        toks = np.array([0, 3, 17, c["T"] - 1])
        s = fp8.token_grads_fp8(L, toks)
        np.testing.assert_allclose(s["dx"], full["dx"][toks], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(s["dgates"], full["dgates"][toks], rtol=1e-11, atol=1e-13)
        cols = np.array([0, 5, c["f"] - 1])
        for e in (0, 3, c["E"] + c["S"] - 1):
            w = fp8.weight_grad_columns_fp8(L, e, cols)
            np.testing.assert_allclose(w["dW_gate"], full["dW_gate"][e][cols], rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(w["dW_up"], full["dW_up"][e][cols], rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(w["dW_down"], full["dW_down"][e][:, cols], rtol=1e-11, atol=1e-12)


# ---- MXFP8 (oracle only)

def test_mx_scales_are_powers_of_two_from_the_block_maximum():
    rng = np.random.default_rng(21)
    v = rng.normal(0, 1, (5, 96)) * np.exp2(rng.integers(-30, 30, (5, 1)))
    v[2, 32:64] = 0.0                                          # an all-zero block
    q, e = fp8.mx_quantize_e4m3(v.astype(np.float32))
    amax = np.abs(v.astype(np.float32).astype(np.float64)).reshape(5, 3, 32).max(axis=2)
    nz = amax > 0
    # 256 <= amax / 2^e < 512 for every non-zero block: e = floor(log2 amax) - 8
    r = amax[nz] / np.ldexp(1.0, e[nz])
    assert np.all((r >= 256) & (r < 512))
    assert e[2, 1] == -127 and not q[2, 32:64].any()


def test_mx_blocks_are_independent_and_lossless_on_the_grid():
    # a block whose values are E4M3 grid values times 2^k with its maximum in [256, 448] * 2^k is
    # exact; changing another block leaves this block's codes and exponent alone
    rng = np.random.default_rng(22)
    grid = fp8.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    grid = grid[grid >= 2.0 ** -3]
    v = rng.choice(grid, (4, 64)) * rng.choice([-1.0, 1.0], (4, 64))
    v[:, 0] = 448.0
    v[:, 32] = 320.0
    v = v * np.exp2(rng.integers(-20, 20, (4, 1)))
    q, e = fp8.mx_quantize_e4m3(v.astype(np.float32))
    assert np.array_equal(fp8.mx_dequantize(q, e), v)
    w = v.copy()
    w[:, 32:] *= 2.0 ** 40
    q2, e2 = fp8.mx_quantize_e4m3(w.astype(np.float32))
    assert np.array_equal(q2[:, :32], q[:, :32]) and np.array_equal(e2[:, 0], e[:, 0])
    assert np.array_equal(e2[:, 1], e[:, 1] + 40)


def test_mx_block_top_saturates():
    # amax just below 512 * 2^k: the block maximum saturates to 448 * 2^k (the format's known
    # clipping), the rest of the block keeps its relative precision
    v = np.full((1, 32), 3.0)
    v[0, 0] = 500.0
    q, e = fp8.mx_quantize_e4m3(v.astype(np.float32))
    d = fp8.mx_dequantize(q, e)
    assert e[0, 0] == 0 and d[0, 0] == 448.0 and np.all(d[0, 1:] == 3.0)


def test_mx_matmul_is_the_product_of_the_dequantised_blocks():
    rng = np.random.default_rng(23)
    a = rng.normal(0, 1, (7, 128))
    b = rng.normal(0, 1, (9, 128)) * np.exp2(rng.integers(-10, 10, (9, 1)))
    aq, ae = fp8.mx_quantize_e4m3(a.astype(np.float32))
    bq, be = fp8.mx_quantize_e4m3(b.astype(np.float32))
    got = fp8.mx_matmul(aq, ae, bq, be)
    # the same sum taken block by block, each block's partial product scaled by both exponents
    ref = np.zeros((7, 9))
    for blk in range(4):
        sl = slice(32 * blk, 32 * blk + 32)
        part = fp8.e4m3_decode(aq[:, sl]) @ fp8.e4m3_decode(bq[:, sl]).T
        ref += part * np.ldexp(1.0, ae[:, blk])[:, None] * np.ldexp(1.0, be[:, blk])[None, :]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-300)
    rel = np.linalg.norm(got - a @ b.T) / np.linalg.norm(a @ b.T)
    assert 1e-3 < rel < 0.1   # e4m3 rounding of both operands, and block maxima clipped at 448
