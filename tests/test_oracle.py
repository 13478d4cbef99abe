"""Pins of the fp64 oracle against things other than itself (CPU only).

* closed forms: routing on logits ln(n_e) (softmax = ratios of integers), a scalar SwiGLU expert,
  the capacity formula;
* a hand-worked dispatch example and a brute-force restatement of queue positions;
* an independent sort-based top-k (the oracle selects by the O(E^2) rank definition);
* invariants: counts sum to T*k, the permutation is a bijection and stable, identity-expert
  combine gives the gate-weighted input, renormalised gates sum to 1;
* E = 1, k = 1 reduces the layer to a dense SwiGLU MLP, checked against scalar loops;
* central finite differences of every input and weight element on a T = 8 instance;
* the sampled (per-token / per-hidden-unit) forms agree with the full pass.
"""
import math
import os

import numpy as np
import pytest

import oracle
import synth


# ------------------------------------------------------------------------------------------
# routing
# ------------------------------------------------------------------------------------------

# logits ln(n_e) => p_e = n_e / sum(n): (n, k, idx, gates as (num, den), renormalised gates)
ROUTING_CASES = [
    ([1, 2, 3, 4], 2, [3, 2], [(4, 10), (3, 10)], [(4, 7), (3, 7)]),
    ([2, 5, 5, 1], 2, [1, 2], [(5, 13), (5, 13)], [(1, 2), (1, 2)]),
    ([2, 5, 5, 1], 1, [1], [(5, 13)], [(1, 1)]),
    ([3, 1, 2], 3, [0, 2, 1], [(3, 6), (2, 6), (1, 6)], [(3, 6), (2, 6), (1, 6)]),
    ([7] * 8, 3, [0, 1, 2], [(1, 8)] * 3, [(1, 3)] * 3),
    ([1, 9, 2, 8, 3, 7], 4, [1, 3, 5, 4], [(9, 30), (8, 30), (7, 30), (3, 30)],
     [(9, 27), (8, 27), (7, 27), (3, 27)]),
]


@pytest.mark.parametrize("n,k,idx,gates,gates_rn", ROUTING_CASES)
def test_routing_closed_form(n, k, idx, gates, gates_rn):
    L = np.log(np.array([n], dtype=np.float64))
    got = oracle.topk_by_rank(L, k)
    assert got.tolist() == [idx]
    p = oracle.softmax(L)
    np.testing.assert_allclose(p[0], np.array(n) / sum(n), rtol=1e-14)
    g = oracle.gates_of(p, got, renorm=False)[0]
    np.testing.assert_allclose(g, [a / b for a, b in gates], rtol=1e-14)
    g = oracle.gates_of(p, got, renorm=True)[0]
    np.testing.assert_allclose(g, [a / b for a, b in gates_rn], rtol=1e-14)


def _topk_by_sort(L, k):
    """Independent top-k: lexicographic sort on (-logit, expert index)."""
    T, E = L.shape
    out = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        order = np.lexsort((np.arange(E), -L[t]))
        out[t] = order[:k]
    return out


@pytest.mark.parametrize("E,k", [(8, 2), (64, 6), (128, 8), (5, 5), (1, 1)])
def test_topk_rank_vs_sort(E, k):
    rng = np.random.default_rng(E * 100 + k)
    L = rng.standard_normal((300, E))
    # plant exact ties: copy some logits onto other experts, and quantise some rows
    L[::7, E // 2] = L[::7, 0]
    L[::5] = np.round(L[::5] * 2) / 2
    assert np.array_equal(oracle.topk_by_rank(L, k), _topk_by_sort(L, k))


def test_gates_sum_rules():
    rng = np.random.default_rng(3)
    L = rng.standard_normal((200, 16)) * 3
    p = oracle.softmax(L)
    idx = oracle.topk_by_rank(L, 4)
    g = oracle.gates_of(p, idx, renorm=False)
    assert np.all(g.sum(1) <= 1 + 1e-15) and np.all(g > 0)
    assert np.all(np.diff(g, axis=1) <= 0)             # slot order = descending logit
    gr = oracle.gates_of(p, idx, renorm=True)
    np.testing.assert_allclose(gr.sum(1), 1.0, rtol=1e-14)
    # renormalised gates equal a softmax taken over the selected logits only
    Ls = np.take_along_axis(L, idx.astype(np.int64), 1)
    np.testing.assert_allclose(gr, oracle.softmax(Ls), rtol=1e-13)


def test_topk_gaps():
    L = np.array([[0.0, 3.0, 1.0, 1.0005]])
    gaps = oracle.topk_gaps(L, 2)
    np.testing.assert_allclose(gaps[0], [3.0 - 1.0005, 0.0005], rtol=1e-12)


# ------------------------------------------------------------------------------------------
# capacity and dispatch
# ------------------------------------------------------------------------------------------

def test_capacity_formula():
    assert oracle.capacity_of(65536, 4, 128, 1.25) == 2560       # GPT-OSS-like workload
    assert oracle.capacity_of(10, 3, 4, 1.0) == 8                # ceil(7.5)
    assert oracle.capacity_of(8, 2, 4, 0.5) == 2
    assert oracle.capacity_of(8, 2, 4, 0.0) is None


def test_dispatch_hand_example():
    idx = np.array([[0, 1], [1, 2], [0, 2], [1, 0], [2, 1]], dtype=np.int32)
    D = oracle.dispatch(idx, 3, None)
    assert D.counts.tolist() == [3, 4, 3]
    assert D.offsets.tolist() == [0, 3, 7, 10]
    assert D.row_of_slot.tolist() == [[0, 3], [4, 7], [1, 8], [5, 2], [9, 6]]
    assert D.token_of_row.tolist() == [0, 2, 3, 0, 1, 3, 4, 1, 2, 4]
    D = oracle.dispatch(idx, 3, 2)
    assert D.counts.tolist() == [3, 4, 3]
    assert D.kept.tolist() == [2, 2, 2]
    assert D.offsets.tolist() == [0, 2, 4, 6]
    assert D.row_of_slot.tolist() == [[0, 2], [3, 4], [1, 5], [-1, -1], [-1, -1]]
    assert D.token_of_row.tolist() == [0, 2, 0, 1, 1, 2]


@pytest.mark.parametrize("T,E,k,C,skew", [(300, 8, 2, None, 0.0), (257, 16, 4, 40, 0.0),
                                          (200, 12, 3, 30, 1.2), (64, 4, 4, None, 0.0),
                                          (50, 6, 1, 3, 2.0)])
def test_dispatch_brute_force(T, E, k, C, skew):
    idx = synth.random_assignments(T + E, T, E, k, skew)
    D = oracle.dispatch(idx, E, C)
    flat = idx.reshape(-1)
    # position of (t, j) = number of earlier assignments (row-major) to the same expert
    pos = np.array([np.count_nonzero(flat[:i] == flat[i]) for i in range(flat.size)])
    assert np.array_equal(D.position.reshape(-1), pos)
    assert D.counts.sum() == T * k
    assert np.array_equal(D.counts, np.bincount(flat, minlength=E))
    kept = D.counts if C is None else np.minimum(D.counts, C)
    assert np.array_equal(D.kept, kept)
    assert np.array_equal(D.offsets, np.concatenate([[0], np.cumsum(kept)]))
    rows = D.row_of_slot.reshape(-1)
    live = rows >= 0
    assert live.sum() == D.offsets[-1]
    assert np.array_equal(np.sort(rows[live]), np.arange(D.offsets[-1]))   # bijection
    # token_of_row inverts row_of_slot, and is non-decreasing within each expert (stable)
    t_of_slot = np.repeat(np.arange(T), k)
    assert np.array_equal(D.token_of_row[rows[live]], t_of_slot[live])
    for e in range(E):
        seg = D.token_of_row[D.offsets[e]:D.offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)
        # kept slots are exactly the first kept[e] in token order
        mine = np.flatnonzero(flat == e)
        assert np.array_equal(np.sort(rows[mine[:kept[e]]]), np.arange(D.offsets[e], D.offsets[e + 1]))
        assert np.all(rows[mine[kept[e]:]] == -1)


# ------------------------------------------------------------------------------------------
# expert FFN and combine
# ------------------------------------------------------------------------------------------

def test_swiglu_scalar_closed_form():
    # d = f = 1: x = 1, W_gate = 2, W_up = 3, W_down = 1/2, upstream dy = 1, gate 1
    x = np.array([[1.0]])
    Wg, Wu, Wd = np.array([[2.0]]), np.array([[3.0]]), np.array([[0.5]])
    s2 = 1.0 / (1.0 + math.exp(-2.0))        # sigma(2)
    a, b, h, o = oracle.expert_forward(x, Wg, Wu, Wd)
    assert a[0, 0] == 2.0 and b[0, 0] == 3.0
    assert abs(h[0, 0] - 3 * 2 * s2) < 1e-14                 # silu(2) * 3, silu(2) = 2 sigma(2)
    assert abs(o[0, 0] - 1.5 * 2 * s2) < 1e-14
    dx, dWg, dWu, dWd, dg = oracle.expert_backward(x, np.array([[1.0]]), np.array([1.0]), Wg, Wu, Wd)
    da = 0.5 * 3 * s2 * (1 + 2 * (1 - s2))   # dh * b * silu'(2), dh = W_down * dy = 1/2
    db = 0.5 * 2 * s2                        # dh * silu(2)
    assert abs(dWg[0, 0] - da) < 1e-14 and abs(dWu[0, 0] - db) < 1e-14
    assert abs(dWd[0, 0] - 3 * 2 * s2) < 1e-14
    assert abs(dx[0, 0] - (2 * da + 3 * db)) < 1e-14
    assert abs(dg[0] - 1.5 * 2 * s2) < 1e-14


def _dense_swiglu_loops(x, Wg, Wu, Wd):
    """Scalar loops: y[t][i] = sum_c Wd[i][c] * silu(sum_m Wg[c][m] x[t][m]) * sum_m Wu[c][m] x[t][m]."""
    T, d = x.shape
    f = Wg.shape[0]
    y = np.zeros((T, d))
    for t in range(T):
        h = []
        for c in range(f):
            a = sum(Wg[c][m] * x[t][m] for m in range(d))
            b = sum(Wu[c][m] * x[t][m] for m in range(d))
            h.append(a / (1.0 + math.exp(-a)) * b)
        for i in range(d):
            y[t][i] = sum(Wd[i][c] * h[c] for c in range(f))
    return y


def _float_inputs(T, d, E, k, f, S, seed, bias=False):
    cfg = dict(T=T, d=d, E=E, k=k, f=f, S=S, renorm=0, cf=0.0, zipf=False)
    G = E + S
    inp = dict(
        x=synth.normal_f32(seed, "x", (T, d), 1.0).astype(np.float64),
        W_r=synth.normal_f32(seed, "W_r", (d, E), 1.0 / math.sqrt(d)).astype(np.float64),
        b_r=(synth.normal_f32(seed, "aux", (E,), 0.5).astype(np.float64) if bias else None),
        W_gate=synth.normal_f32(seed, "W_gate", (G, f, d), 1.0 / math.sqrt(d)).astype(np.float64),
        W_up=synth.normal_f32(seed, "W_up", (G, f, d), 1.0 / math.sqrt(d)).astype(np.float64),
        W_down=synth.normal_f32(seed, "W_down", (G, d, f), 1.0 / math.sqrt(f)).astype(np.float64),
        dy=synth.normal_f32(seed, "dy", (T, d), 1.0).astype(np.float64),
    )
    return cfg, inp


def test_single_expert_is_dense_swiglu():
    cfg, inp = _float_inputs(T=5, d=6, E=1, k=1, f=7, S=0, seed=11)
    y, _ = oracle.Layer(inp, cfg).forward()
    ref = _dense_swiglu_loops(inp["x"], inp["W_gate"][0], inp["W_up"][0], inp["W_down"][0])
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)


def test_shared_experts_add_dense_swiglu():
    cfg, inp = _float_inputs(T=6, d=5, E=3, k=1, f=4, S=2, seed=12)
    L1 = oracle.Layer(inp, cfg)
    y, o_slot = L1.forward()
    R = L1.routing()
    routed = R.gates[:, 0:1] * o_slot[:, 0]
    shared = sum(_dense_swiglu_loops(inp["x"], inp["W_gate"][3 + s], inp["W_up"][3 + s],
                                     inp["W_down"][3 + s]) for s in range(2))
    np.testing.assert_allclose(y, routed + shared, rtol=1e-12, atol=1e-13)
    # routed part: the selected expert's dense SwiGLU, weighted by its gate
    for t in range(6):
        e = R.idx[t, 0]
        ref = _dense_swiglu_loops(inp["x"][t:t + 1], inp["W_gate"][e], inp["W_up"][e], inp["W_down"][e])
        np.testing.assert_allclose(o_slot[t, 0], ref[0], rtol=1e-12, atol=1e-13)


def test_identity_expert_combine():
    rng = np.random.default_rng(5)
    T, k, d = 40, 3, 8
    x = rng.standard_normal((T, d))
    g = rng.random((T, k))
    kept = rng.random((T, k)) > 0.3
    o_slot = np.repeat(x[:, None, :], k, axis=1)          # every expert is the identity
    y = oracle.combine(o_slot, g, kept)
    np.testing.assert_allclose(y, (g * kept).sum(1)[:, None] * x, rtol=1e-14)


# ------------------------------------------------------------------------------------------
# gradients: central differences on a T = 8 instance, every element of every input
# ------------------------------------------------------------------------------------------

FD_CASES = {
    "plain": dict(renorm=0, cf=0.0, S=0, bias=False),
    "renorm_shared_bias": dict(renorm=1, cf=0.0, S=2, bias=True),
    "capacity_drops": dict(renorm=0, cf=0.5, S=0, bias=False),
    "capacity_renorm_shared": dict(renorm=1, cf=0.75, S=1, bias=True),
}


@pytest.mark.parametrize("case", list(FD_CASES))
def test_finite_differences(case):
    c = FD_CASES[case]
    cfg, inp = _float_inputs(T=8, d=16, E=4, k=2, f=32, S=c["S"], seed=21, bias=c["bias"])
    cfg.update(renorm=c["renorm"], cf=c["cf"])
    L0 = oracle.Layer(inp, cfg)
    grads = L0.backward()
    idx0 = L0.routing().idx
    disp0 = L0.dispatch()
    if c["cf"] > 0:
        assert np.any(disp0.row_of_slot < 0), "case meant to drop slots"
    dy = inp["dy"]

    def loss(pert):
        Lp = oracle.Layer(pert, cfg)
        y, _ = Lp.forward()
        assert np.array_equal(Lp.routing().idx, idx0), "perturbation flipped the selection"
        return float(np.sum(dy * y))

    h = 1e-6
    names = {"x": "dx", "W_r": "dW_r", "W_gate": "dW_gate", "W_up": "dW_up", "W_down": "dW_down"}
    if c["bias"]:
        names["b_r"] = "db_r"
    for name, gname in names.items():
        base = inp[name]
        an = grads[gname]
        fd = np.zeros_like(base)
        for i in np.ndindex(base.shape):
            p = dict(inp)
            arr = base.copy()
            arr[i] += h
            p[name] = arr
            lp = loss(p)
            arr[i] -= 2 * h
            lm = loss(p)
            fd[i] = (lp - lm) / (2 * h)
        scale = np.max(np.abs(an))
        assert scale > 0
        err = np.max(np.abs(fd - an))
        assert err <= 1e-6 * scale, (name, err, scale)


def test_dgates_are_dy_dot_expert_output():
    cfg, inp = _float_inputs(T=8, d=16, E=4, k=2, f=32, S=0, seed=22)
    cfg["cf"] = 0.5
    L = oracle.Layer(inp, cfg)
    _, o_slot = L.forward()
    g = L.backward()
    kept = L.dispatch().row_of_slot >= 0
    ref = np.einsum("td,tjd->tj", inp["dy"], o_slot) * kept
    np.testing.assert_allclose(g["dgates"], ref, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------------------------------
# sampled forms used for full-size workloads
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("renorm,cf,S", [(0, 0.0, 0), (1, 0.0, 2), (0, 1.0, 0)])
def test_sampled_forms_match_full(renorm, cf, S):
    cfg = dict(T=96, d=64, E=8, k=2, f=128, S=S, renorm=renorm, cf=cf, zipf=False)
    inp = synth.make_inputs(cfg, seed=4)
    if cf > 0:
        inp["b_r"] = synth.zipf_bias(4, 8)          # skew so the capacity drops slots
    L = oracle.Layer(inp, cfg)
    y, _ = L.forward()
    full = L.backward()
    if cf > 0:
        assert np.any(L.dispatch().row_of_slot < 0)
    toks = np.array([0, 5, 17, 95, 42])
    s = L.token_outputs(toks)
    np.testing.assert_allclose(s["y"], y[toks], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(s["dx"], full["dx"][toks], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(s["dgates"], full["dgates"][toks], rtol=1e-11, atol=1e-13)
    for e in [0, 3, 7] + ([8, 9] if S else []):
        cols = np.array([0, 7, 127])
        w = L.weight_grad_columns(e, cols)
        np.testing.assert_allclose(w["dW_gate"], full["dW_gate"][e][cols], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(w["dW_up"], full["dW_up"][e][cols], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(w["dW_down"], full["dW_down"][e][:, cols], rtol=1e-11, atol=1e-12)


# ------------------------------------------------------------------------------------------
# rounding to bf16 (the value a bf16 intermediate holds)
# ------------------------------------------------------------------------------------------

def _bf16_grid():
    """Every finite non-negative bf16 value with its bit pattern, plus 2^128 standing for the
    overflow to infinity (its pattern 0x7F80 is even, as round-to-nearest-even treats it)."""
    bits = np.arange(0, 0x7F81, dtype=np.uint32)
    vals = (bits << np.uint32(16)).view(np.float32).astype(np.float64)
    vals[-1] = 2.0 ** 128
    return bits, vals


def _bf16_brute(v: float) -> float:
    """Nearest grid value by exact rational distances; a tie takes the even bit pattern."""
    from fractions import Fraction
    if v != v or v in (math.inf, -math.inf):
        return v
    bits, vals = _bf16_grid()
    a = abs(v)
    i = int(np.searchsorted(vals, a))                     # vals[i-1] < a <= vals[i]
    cands = [j for j in (i - 1, i) if 0 <= j < len(vals)]
    fa = Fraction(a)
    dist = [abs(Fraction(vals[j]) - fa) for j in cands]
    best = min(dist)
    pick = [j for j, dd in zip(cands, dist) if dd == best]
    j = pick[0] if len(pick) == 1 else [p for p in pick if bits[p] % 2 == 0][0]
    r = math.inf if j == len(vals) - 1 else vals[j]
    return math.copysign(r, v)


def test_bf16_rounding_hand_cases():
    one = 1.0
    cases = [
        (one + 2.0 ** -8, 1.0),                            # tie between 1 and 1 + 2^-7: even (1)
        (one + 3 * 2.0 ** -8, one + 2.0 ** -6),            # tie between odd and even: up to even
        (one + 2.0 ** -8 + 2.0 ** -40, one + 2.0 ** -7),   # just above a tie (lost by a float32 step)
        (one + 2.0 ** -8 - 2.0 ** -40, 1.0),               # just below it
        (2.0 - 2.0 ** -9, 2.0),                            # just below a binade rounds into it
        (2.0 - 2.0 ** -8 - 2.0 ** -30, 2.0 - 2.0 ** -7),
        (-(one + 3 * 2.0 ** -8), -(one + 2.0 ** -6)),      # sign symmetric
        (0.0, 0.0), (-0.0, -0.0),
        (oracle.moe_oracle.BF16_MAX, oracle.moe_oracle.BF16_MAX),
        (oracle.moe_oracle.BF16_MAX + 2.0 ** 118, oracle.moe_oracle.BF16_MAX),   # below the halfway point
        (oracle.moe_oracle.BF16_MAX + 2.0 ** 119, math.inf),                     # halfway: to even = overflow
        (-1e39, -math.inf), (1e300, math.inf),
        (2.0 ** -133, 2.0 ** -133),                        # smallest subnormal
        (2.0 ** -134, 0.0),                                # half of it: tie to even (zero)
        (3 * 2.0 ** -134, 2.0 ** -132),                    # 1.5 steps: tie to even (2 steps)
        (-2.0 ** -140, -0.0),
        (2.0 ** -126 - 2.0 ** -134, 2.0 ** -126),          # top of the subnormals rounds to the min normal
        (math.inf, math.inf), (-math.inf, -math.inf),
    ]
    got = oracle.f64_to_bf16_value(np.array([c[0] for c in cases]))
    for (v, want), g in zip(cases, got):
        assert g == want and math.copysign(1, g) == math.copysign(1, want), (v, g, want)
    assert np.isnan(oracle.f64_to_bf16_value(np.array([math.nan]))[0])


def test_bf16_rounding_brute_force():
    rng = np.random.default_rng(5)
    v = rng.normal(size=400) * np.exp2(rng.integers(-140, 130, 400))
    # exact ties of the bf16 grid and one float64 ulp either side of them
    base = synth.bf16_bits_to_f32(rng.integers(0, 0x7F7F, 100).astype(np.uint16)).astype(np.float64)
    base = base[base > 2.0 ** -120]
    _, e = np.frexp(base)
    tie = base + np.ldexp(1.0, e - 9)                      # half a bf16 step above a grid value
    v = np.concatenate([v, tie, np.nextafter(tie, 0), np.nextafter(tie, np.inf), -tie])
    got = oracle.f64_to_bf16_value(v)
    want = np.array([_bf16_brute(float(a)) for a in v])
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_bf16_rounding_matches_torch_on_float32_inputs():
    """On values that float32 holds exactly, torch's float32 -> bfloat16 conversion (round to
    nearest even) is one rounding too, so both must agree bit for bit."""
    import torch
    rng = np.random.default_rng(6)
    u = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    u[:2000] = (u[:2000] & np.uint32(0xFFFF0000)) | np.uint32(0x8000)   # exact ties
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.f64_to_bf16_value(f.astype(np.float64))
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_stored_summary_of_tiny_workload():
    """Regression guard: the oracle's tiny-workload results, written by tests/golden/make_golden.py."""
    import json
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_oracle_summary.json")
    ref = json.load(open(path))
    from golden.make_golden import summarise
    got = summarise()
    assert got["counts"] == ref["counts"]
    assert got["idx_head"] == ref["idx_head"]
    for key in ("fp8_x_codes_head", "fp8_x_scales_head", "mx_x_codes_head", "mx_x_exps"):
        assert got[key] == ref[key], key
    for key in ref["norms"]:
        assert abs(got["norms"][key] - ref["norms"][key]) <= 1e-12 * abs(ref["norms"][key]), key
