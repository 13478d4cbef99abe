"""fp64 CPU oracle of the single-GPU Mixture-of-Experts SwiGLU FFN layer, forward and backward.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this module.  The product path (``mixture_experts_layer_10_gb300``) never
calls it, and the two share no code: this file widens bf16 itself, computes in float64
throughout, and uses only numpy (``@`` matmul, ``exp``, sums) as library primitives.  There is no
blocking, fusion or reordering here beyond what each definition states.

What the pages fix and what they leave open
-------------------------------------------
The pages describe MoE training systems, not the layer's formulas:

* "Piper: Efficient Large-Scale MoE Training via Resource Modeling and Pipelined Hybrid
  Parallelism" (Japanese explainer, section "the problem"): a router picks a few experts for
  each token and the rest stay idle; load can be badly skewed towards one expert.
* "MoEBlaze: Breaking the Memory Wall for Efficient MoE Training on Modern GPUs" (Korean
  summary), Methodology item 1: tokens go to experts through compact per-expert dispatch
  queues built on the fly, with no dense token-by-expert routing matrix; item 2: fused
  scatter-gather (dispatch / reverse dispatch) around the expert feed-forward, and selective
  activation checkpointing that stores a minimum and recomputes the rest in backward;
  "Limitations": a static top-k routing policy.
* "DisagMoE" technical summary, section 2.2: dispatch and combine around the expert FFN.

Everything else is the plainest standard reading, taken as follows (each is repeated at the
function that uses it):

1. logits = x W_r + b (b only when a router bias is given).
2. p = softmax(logits) over all E routed experts; experts are selected by logit, top-k,
   larger logit first, a tie going to the lower expert index; slot j holds the j-th best.
3. gate g_j = p[idx_j]; with renormalisation g_j = p[idx_j] / sum_m p[idx_m].
4. per-expert capacity C = ceil(cf*T*k/E) (none when cf <= 0): within each expert the
   assignments are taken in token order (t, then slot j) and those at position >= C are dropped;
   dropped slots contribute nothing and get a zero gate gradient.
5. expert e: a = W_gate[e] x, b = W_up[e] x, h = silu(a)*b with silu(z) = z/(1+exp(-z)),
   o = W_down[e] h; no biases.
6. shared experts (indices E..E+S-1) see every token with weight 1, outside softmax/top-k.
7. y_t = sum over kept slots g_j o_{t,j} + sum_s o^s_t.
8. the backward is the exact derivative of 1-7, with top-k selection and drops held fixed.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


# --------------------------------------------------------------------------------------------
# input widening (the oracle's own; bf16 values are stored as raw uint16 bits)
# --------------------------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 bits: the bf16 pattern is the top half of an fp32 pattern."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def as_f64(a) -> np.ndarray:
    """bf16 bits (uint16) are widened exactly; any float array is taken as its float64 value."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return bf16_to_f64(a)
    return a.astype(np.float64)


BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127     # largest finite bf16


def f64_to_bf16_value(v: np.ndarray) -> np.ndarray:
    """The value of ``v`` rounded once to bf16 (nearest, ties to even), returned as float64.

    bf16 keeps 8 significant bits and fp32's exponent range: a value whose leading bit is
    2^p (p >= -126) is rounded to a multiple of 2^(p-7); below 2^-126 the step stays 2^-133
    (subnormals).  The rounding is done directly from float64 (no float32 step, which would
    round twice), with numpy's rint (half to even) on the scaled value.  Magnitudes that round
    above the largest finite bf16 become infinities; zeros keep their sign; inf and nan pass.
    """
    a = np.asarray(v, dtype=np.float64)
    out = a.copy()
    fin = np.isfinite(a)
    mag = np.abs(a[fin])
    _, e = np.frexp(mag)                                   # mag = m 2^e, m in [0.5, 1)
    q = np.maximum(e - 1, -126) - 7                        # exponent of the rounding step
    r = np.ldexp(np.rint(np.ldexp(mag, -q)), q)
    r = np.where(r > BF16_MAX, np.inf, r)
    out[fin] = np.copysign(r, a[fin])
    return out


def capacity_of(T: int, k: int, E: int, cf: float) -> int | None:
    """Reading 4: C = ceil(cf*T*k/E), or None (no capacity, dropless) when cf <= 0."""
    if cf is None or cf <= 0:
        return None
    return int(math.ceil(cf * T * k / E))


# --------------------------------------------------------------------------------------------
# routing: readings 1-3
# --------------------------------------------------------------------------------------------

def router_logits(x: np.ndarray, W_r: np.ndarray, b_r: np.ndarray | None) -> np.ndarray:
    """Reading 1: logits[t,e] = sum_i x[t,i] W_r[i,e] (+ b[e]), in float64."""
    logits = np.asarray(x, np.float64) @ np.asarray(W_r, np.float64)
    if b_r is not None:
        logits = logits + np.asarray(b_r, np.float64)[None, :]
    return logits


def topk_by_rank(logits: np.ndarray, k: int) -> np.ndarray:
    """Reading 2, stated as a definition: expert e has rank
        rank_e = #{e' : l_e' > l_e  or  (l_e' == l_e and e' < e)},
    it is selected iff rank_e < k, and it goes to slot rank_e.  O(E^2) per token.
    Returns idx [T,k] int32.
    """
    L = np.asarray(logits, np.float64)
    T, E = L.shape
    idx = np.empty((T, k), dtype=np.int32)
    lower = np.arange(E)[None, :] < np.arange(E)[:, None]     # lower[e, e'] = e' < e
    step = max(1, (1 << 22) // (E * E))
    for t0 in range(0, T, step):
        blk = L[t0:t0 + step]                                  # [b, E]
        le = blk[:, :, None]                                   # l_e
        lp = blk[:, None, :]                                   # l_e'
        beats = (lp > le) | ((lp == le) & lower[None, :, :])
        rank = beats.sum(axis=2)                               # [b, E]
        tt, ee = np.nonzero(rank < k)                          # selected (token, expert)
        idx[t0 + tt, rank[tt, ee]] = ee
    return idx


def softmax(logits: np.ndarray) -> np.ndarray:
    """Reading 2: p = exp(l - max l) / sum exp(l - max l) over the E routed experts."""
    L = np.asarray(logits, np.float64)
    z = np.exp(L - L.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def gates_of(p: np.ndarray, idx: np.ndarray, renorm: bool) -> np.ndarray:
    """Reading 3: g_j = p[idx_j], or p[idx_j] / sum_m p[idx_m] when renormalised."""
    g = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    if renorm:
        g = g / g.sum(axis=1, keepdims=True)
    return g


@dataclass
class Routing:
    logits: np.ndarray   # [T,E] f64
    p: np.ndarray        # [T,E] f64
    idx: np.ndarray      # [T,k] int32
    gates: np.ndarray    # [T,k] f64


def route(x: np.ndarray, W_r: np.ndarray, b_r, k: int, renorm: bool) -> Routing:
    L = router_logits(x, W_r, b_r)
    p = softmax(L)
    idx = topk_by_rank(L, k)
    return Routing(L, p, idx, gates_of(p, idx, renorm))


def topk_gaps(logits: np.ndarray, k: int) -> np.ndarray:
    """Sorted-logit gaps of each token: column j is l_(j) - l_(j+1) for j < min(k, E-1).

    Column k-1 is the k-th vs (k+1)-th gap that decides the selected set; the earlier columns
    decide the slot order.  Missing gaps (k == E) are +inf.
    """
    L = -np.sort(-np.asarray(logits, np.float64), axis=1)
    T, E = L.shape
    gaps = np.full((T, k), np.inf)
    for j in range(min(k, E - 1)):
        gaps[:, j] = L[:, j] - L[:, j + 1]
    return gaps


# --------------------------------------------------------------------------------------------
# dispatch queues (MoEBlaze, Methodology item 1) and capacity (reading 4)
# --------------------------------------------------------------------------------------------

@dataclass
class Dispatch:
    counts: np.ndarray        # [E] raw demand per expert; sums to T*k
    kept: np.ndarray          # [E] min(counts, C)
    offsets: np.ndarray       # [E+1] exclusive scan of kept; offsets[E] = rows kept
    position: np.ndarray      # [T,k] position of the slot in its expert's queue (token order)
    row_of_slot: np.ndarray   # [T,k] offsets[e] + position, or -1 when dropped
    token_of_row: np.ndarray  # [offsets[E]] token of each kept row
    slot_of_row: np.ndarray   # [offsets[E]] flat slot t*k+j of each kept row


def dispatch(idx: np.ndarray, E: int, C: int | None) -> Dispatch:
    """Per-expert queues in token order, with no T x E matrix.

    Walk the assignments (t, j) in row-major order and append each to its expert's queue;
    the queue position is its rank.  counts = queue lengths, kept = min(counts, C),
    offsets = exclusive scan of kept, row = offsets[e] + position for kept slots.
    """
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    position = np.zeros((T, k), dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            position[t, j] = counts[e]
            counts[e] += 1
    kept = counts.copy() if C is None else np.minimum(counts, C)
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + kept[e]
    n = int(offsets[E])
    row_of_slot = np.full((T, k), -1, dtype=np.int64)
    token_of_row = np.full(n, -1, dtype=np.int64)
    slot_of_row = np.full(n, -1, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            if position[t, j] < kept[e]:
                r = int(offsets[e] + position[t, j])
                row_of_slot[t, j] = r
                token_of_row[r] = t
                slot_of_row[r] = t * k + j
    return Dispatch(counts, kept, offsets, position, row_of_slot, token_of_row, slot_of_row)


# --------------------------------------------------------------------------------------------
# expert SwiGLU FFN: reading 5
# --------------------------------------------------------------------------------------------

def silu(z):
    return z / (1.0 + np.exp(-z))


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def expert_forward(xr, Wg, Wu, Wd):
    """Rows xr [n,d] through one expert: a = xr Wg^T, b = xr Wu^T, h = silu(a) b, o = h Wd^T."""
    a = xr @ Wg.T
    b = xr @ Wu.T
    h = silu(a) * b
    o = h @ Wd.T
    return a, b, h, o


def expert_backward(xr, dyr, g, Wg, Wu, Wd):
    """Exact derivative of g * expert(xr) for rows xr with upstream dyr and per-row weight g.

    Returns dxr, dWg, dWu, dWd and dg (the gradient of each row's gate, dy . o).
      do  = g dy;      dh = do Wd;      dWd = do^T h
      da  = dh * b * sigma(a) * (1 + a (1 - sigma(a)));   db = dh * silu(a)
      dWg = da^T xr;   dWu = db^T xr;   dxr = da Wg + db Wu
    """
    a, b, h, o = expert_forward(xr, Wg, Wu, Wd)
    s = sigmoid(a)
    do = g[:, None] * dyr
    dh = do @ Wd
    da = dh * b * s * (1.0 + a * (1.0 - s))
    db = dh * (a * s)
    dWd = do.T @ h
    dWg = da.T @ xr
    dWu = db.T @ xr
    dxr = da @ Wg + db @ Wu
    dg = np.sum(dyr * o, axis=1)
    return dxr, dWg, dWu, dWd, dg


# --------------------------------------------------------------------------------------------
# combine (reverse dispatch): reading 7
# --------------------------------------------------------------------------------------------

def combine(o_slot, gates, kept, shared_o=None):
    """y_t = sum over kept slots j of g_tj o_tj, plus the shared experts' outputs (weight 1).

    o_slot [T,k,d] holds each slot's expert output, kept [T,k] says which slots survived the
    capacity; shared_o is a list of [T,d] outputs of the always-on experts.
    """
    T, k, d = o_slot.shape
    y = np.zeros((T, d))
    for j in range(k):
        w = np.where(kept[:, j], gates[:, j], 0.0)
        y += w[:, None] * o_slot[:, j]
    for os_ in (shared_o or []):
        y += os_
    return y


# --------------------------------------------------------------------------------------------
# router backward: derivative of readings 2-3 with the selection held fixed
# --------------------------------------------------------------------------------------------

def router_backward_logits(p, idx, gates, dgates, renorm: bool):
    """dL/dlogits from dL/dgates.

    Without renormalisation g_j = p[idx_j] and dp_a/dl_b = p_a (delta_ab - p_b), so
        dl_b = p_b * (dg_{j(b)} [b selected] - sum_j dg_j g_j).
    With renormalisation g is the softmax over the selected logits only, so
        dl_{idx_j} = g_j (dg_j - sum_m dg_m g_m), and 0 for experts not selected.
    """
    T, E = p.shape
    k = idx.shape[1]
    s = np.sum(dgates * gates, axis=1)                   # [T]
    dl = np.zeros((T, E))
    if renorm:
        for j in range(k):
            dl[np.arange(T), idx[:, j]] += gates[:, j] * (dgates[:, j] - s)
    else:
        sel = np.zeros((T, E))
        for j in range(k):
            sel[np.arange(T), idx[:, j]] += dgates[:, j]
        dl = p * (sel - s[:, None])
    return dl


def router_backward(x, W_r, dlogits):
    """Through logits = x W_r + b: dW_r = x^T dl, db = sum_t dl_t, dx = dl W_r^T."""
    x = np.asarray(x, np.float64)
    W_r = np.asarray(W_r, np.float64)
    return x.T @ dlogits, dlogits.sum(axis=0), dlogits @ W_r.T


# --------------------------------------------------------------------------------------------
# the whole layer
# --------------------------------------------------------------------------------------------

class Layer:
    """One MoE layer instance: the inputs of one workload, widened to float64 on demand.

    ``inp`` holds x [T,d], W_r [d,E], b_r [E] or None, W_gate/W_up [E+S,f,d], W_down [E+S,d,f]
    and dy [T,d]; bf16 tensors are raw uint16 bits.  ``cfg`` holds T, d, E, k, f, S, renorm, cf.
    """

    def __init__(self, inp: dict, cfg: dict):
        self.inp = inp
        self.cfg = cfg
        self.T, self.d, self.E, self.k = cfg["T"], cfg["d"], cfg["E"], cfg["k"]
        self.f, self.S = cfg["f"], cfg["S"]
        self.renorm = bool(cfg["renorm"])
        self.C = capacity_of(self.T, self.k, self.E, cfg["cf"])
        self._x = None
        self._dy = None
        self._routing = None
        self._disp = None

    # ---- widened inputs
    @property
    def x(self):
        if self._x is None:
            self._x = as_f64(self.inp["x"])
        return self._x

    @property
    def dy(self):
        if self._dy is None:
            self._dy = as_f64(self.inp["dy"])
        return self._dy

    def W(self, g: int):
        """Expert g's (W_gate, W_up, W_down) in float64 (g >= E are the shared experts)."""
        return (as_f64(self.inp["W_gate"][g]), as_f64(self.inp["W_up"][g]),
                as_f64(self.inp["W_down"][g]))

    # ---- routing and dispatch (over all tokens)
    def routing(self, idx: np.ndarray | None = None) -> Routing:
        """Route every token.  ``idx`` may fix the assignment (it must then come from the oracle
        itself or from a test's own input); gates are recomputed in float64 for it."""
        if self._routing is None or idx is not None:
            L = router_logits(self.x, self.inp["W_r"], self.inp.get("b_r"))
            p = softmax(L)
            sel = topk_by_rank(L, self.k) if idx is None else np.asarray(idx, np.int32)
            r = Routing(L, p, sel, gates_of(p, sel, self.renorm))
            if idx is not None:
                return r
            self._routing = r
        return self._routing

    def dispatch(self) -> Dispatch:
        if self._disp is None:
            self._disp = dispatch(self.routing().idx, self.E, self.C)
        return self._disp

    # ---- full forward / backward
    def forward(self):
        """y [T,d] (float64, unrounded) and per-slot expert outputs o [T,k,d] (0 when dropped)."""
        R, D = self.routing(), self.dispatch()
        T, k, d = self.T, self.k, self.d
        o_slot = np.zeros((T, k, d))
        for e in range(self.E):
            rows = np.arange(D.offsets[e], D.offsets[e + 1])
            if rows.size == 0:
                continue
            slots = D.slot_of_row[rows]
            t_of, j_of = slots // k, slots % k
            Wg, Wu, Wd = self.W(e)
            _, _, _, o = expert_forward(self.x[t_of], Wg, Wu, Wd)
            o_slot[t_of, j_of] = o
        shared = [expert_forward(self.x, *self.W(self.E + s))[3] for s in range(self.S)]
        y = combine(o_slot, R.gates, D.row_of_slot >= 0, shared)
        return y, o_slot

    def backward(self):
        """All gradients of sum(dy * y): dx, dW_r, db_r, dW_gate, dW_up, dW_down, dgates, dlogits."""
        R, D = self.routing(), self.dispatch()
        T, k, d, f, E, S = self.T, self.k, self.d, self.f, self.E, self.S
        dx = np.zeros((T, d))
        dW_gate = np.zeros((E + S, f, d))
        dW_up = np.zeros((E + S, f, d))
        dW_down = np.zeros((E + S, d, f))
        dgates = np.zeros((T, k))
        for e in range(E):
            rows = np.arange(D.offsets[e], D.offsets[e + 1])
            if rows.size == 0:
                continue
            slots = D.slot_of_row[rows]
            t_of, j_of = slots // k, slots % k
            Wg, Wu, Wd = self.W(e)
            dxr, dWg, dWu, dWd, dg = expert_backward(self.x[t_of], self.dy[t_of],
                                                     R.gates[t_of, j_of], Wg, Wu, Wd)
            np.add.at(dx, t_of, dxr)
            dW_gate[e], dW_up[e], dW_down[e] = dWg, dWu, dWd
            dgates[t_of, j_of] = dg
        for s in range(S):
            Wg, Wu, Wd = self.W(E + s)
            dxr, dWg, dWu, dWd, _ = expert_backward(self.x, self.dy, np.ones(T), Wg, Wu, Wd)
            dx += dxr
            dW_gate[E + s], dW_up[E + s], dW_down[E + s] = dWg, dWu, dWd
        dl = router_backward_logits(R.p, R.idx, R.gates, dgates, self.renorm)
        dW_r, db_r, dx_r = router_backward(self.x, self.inp["W_r"], dl)
        dx += dx_r
        return dict(dx=dx, dW_r=dW_r, db_r=db_r, dW_gate=dW_gate, dW_up=dW_up,
                    dW_down=dW_down, dgates=dgates, dlogits=dl)

    # ---- sampled forms for workloads too large for a full float64 pass
    def token_outputs(self, tokens: np.ndarray):
        """y[tokens], dx[tokens] and dgates[tokens] computed one token at a time.

        Each token's outputs depend only on its own routing and on whether its slots were
        dropped (which needs the queue positions over all tokens when a capacity is set).
        """
        tokens = np.asarray(tokens, np.int64)
        k, E, S = self.k, self.E, self.S
        if self.C is not None:
            D = self.dispatch()
            R = self.routing()
            L, p, idx, g = R.logits[tokens], R.p[tokens], R.idx[tokens], R.gates[tokens]
            kept = D.row_of_slot[tokens] >= 0
        else:
            xs = self.x[tokens]
            L = router_logits(xs, self.inp["W_r"], self.inp.get("b_r"))
            p = softmax(L)
            idx = topk_by_rank(L, k)
            g = gates_of(p, idx, self.renorm)
            kept = np.ones(idx.shape, dtype=bool)
        n = tokens.size
        xs, dys = self.x[tokens], self.dy[tokens]
        y = np.zeros((n, self.d))
        dx = np.zeros((n, self.d))
        dgates = np.zeros((n, k))
        for e in range(E + S):
            if e < E:
                sel = np.argwhere((idx == e) & kept)            # (token-in-sample, slot)
                if sel.size == 0:
                    continue
                ti, jj = sel[:, 0], sel[:, 1]
                gw = g[ti, jj]
            else:
                ti = np.arange(n)
                jj = None
                gw = np.ones(n)
            Wg, Wu, Wd = self.W(e)
            _, _, _, o = expert_forward(xs[ti], Wg, Wu, Wd)
            dxr, _, _, _, dg = expert_backward(xs[ti], dys[ti], gw, Wg, Wu, Wd)
            np.add.at(y, ti, gw[:, None] * o)
            np.add.at(dx, ti, dxr)
            if jj is not None:
                dgates[ti, jj] = dg
        dl = router_backward_logits(p, idx, g, dgates, self.renorm)
        dx += dl @ np.asarray(self.inp["W_r"], np.float64).T
        return dict(y=y, dx=dx, dgates=dgates, idx=idx, gates=g, logits=L)

    def weight_grad_columns(self, e: int, cols: np.ndarray):
        """dW_gate[e][cols,:], dW_up[e][cols,:] and dW_down[e][:,cols] for hidden units ``cols``.

        Hidden unit c of expert e needs only column c of a, b and dh over the rows routed to e,
        so these entries are exact without the rest of the expert.
        """
        cols = np.asarray(cols, np.int64)
        k = self.k
        if e < self.E:
            D, R = self.dispatch(), self.routing()
            rows = np.arange(D.offsets[e], D.offsets[e + 1])
            slots = D.slot_of_row[rows]
            t_of, j_of = slots // k, slots % k
            gw = R.gates[t_of, j_of]
        else:
            t_of = np.arange(self.T)
            gw = np.ones(self.T)
        Wg, Wu, Wd = self.W(e)
        xr, dyr = self.x[t_of], self.dy[t_of]
        a = xr @ Wg[cols].T
        b = xr @ Wu[cols].T
        s = sigmoid(a)
        h = a * s * b
        do = gw[:, None] * dyr
        dh = do @ Wd[:, cols]
        da = dh * b * s * (1.0 + a * (1.0 - s))
        db = dh * (a * s)
        return dict(dW_gate=da.T @ xr, dW_up=db.T @ xr, dW_down=do.T @ h)
