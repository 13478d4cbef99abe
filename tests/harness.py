"""Helpers shared by the parity tests: tensor conversion, the padded row layout the ABI documents,
and the tolerance rules.

Tolerance rules (one per kind of output):
  * integer / index outputs (idx where the decision is unambiguous, counts, offsets, rows):
    bit-exact;
  * bf16 outputs and all gradients: |err| <= 2e-2 * max|ref| + 1e-2 * |ref| elementwise, with
    max|ref| taken per tensor (per expert for weight gradients);
  * fp32 router gates: relative error <= 1e-5.
"""
from __future__ import annotations

import numpy as np

import oracle

ABS_FRAC = 2e-2
REL = 1e-2
GATE_REL = 1e-5
TIE_GAP = 1e-3


def to_dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_dev(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def from_dev_bf16(t) -> np.ndarray:
    """Device bf16 tensor -> float64 numpy (exact)."""
    import torch
    u = t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return oracle.bf16_to_f64(u)


def from_dev(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def padded_starts(kept: np.ndarray) -> np.ndarray:
    """Segment starts of the documented padded layout: P_0 = 0, P_{g+1} = P_g + roundup(n_g, 256)."""
    P = np.zeros(len(kept) + 1, dtype=np.int64)
    for g, n in enumerate(kept):
        P[g + 1] = P[g] + (int(n) + 255) // 256 * 256
    return P


def segment_rows(D: oracle.Dispatch, T: int, S: int):
    """Per segment (routed then shared): kept row count and padded start, from the oracle's queues."""
    kept = np.concatenate([D.kept, np.full(S, T, dtype=np.int64)])
    return kept, padded_starts(kept)


def check_close(name: str, got: np.ndarray, ref: np.ndarray, max_ref: float | None = None):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite output"
    m = float(np.max(np.abs(ref))) if max_ref is None else max_ref
    err = np.abs(got - ref)
    bound = ABS_FRAC * m + REL * np.abs(ref)
    bad = err > bound
    if np.any(bad):
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{name}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} (max|ref| {m:.4g})")


def check_weight_grad(name: str, got: np.ndarray, ref: np.ndarray):
    """Weight gradients [G, ...]: max|ref| taken per expert, so small experts are not masked."""
    for g in range(ref.shape[0]):
        m = float(np.max(np.abs(ref[g])))
        if m == 0.0:
            assert np.all(got[g] == 0), f"{name}[{g}]: expert without rows must have zero gradient"
        else:
            check_close(f"{name}[{g}]", got[g], ref[g], m)


def check_gates(got: np.ndarray, ref: np.ndarray, mask: np.ndarray | None = None):
    got = np.asarray(got, np.float64)
    rel = np.abs(got - ref) / np.abs(ref)
    if mask is not None:
        rel = rel[mask]
    assert rel.size == 0 or rel.max() <= GATE_REL, f"gates: worst relative error {rel.max():.3e}"


def decided_tokens(logits: np.ndarray, k: int):
    """Tokens whose top-k set and slot order are both decided by gaps above the tie threshold,
    and tokens whose set (only) is decided."""
    gaps = oracle.topk_gaps(logits, k)
    set_ok = gaps[:, k - 1] > TIE_GAP
    order_ok = set_ok & np.all(gaps[:, :k - 1] > TIE_GAP, axis=1) if k > 1 else set_ok
    return order_ok, set_ok


def check_routing(idx_gpu: np.ndarray, gates_gpu: np.ndarray, R: oracle.Routing, k: int):
    """Rule: idx bit-exact where decided; elsewhere the GPU's choice must be a valid top-k within
    the tie threshold.  Gates within 1e-5 relative on tokens whose idx matches."""
    order_ok, set_ok = decided_tokens(R.logits, k)
    assert np.array_equal(idx_gpu[order_ok], R.idx[order_ok]), "top-k order mismatch on decided tokens"
    assert np.array_equal(np.sort(idx_gpu[set_ok], 1), np.sort(R.idx[set_ok], 1)), "top-k set mismatch"
    # undecided tokens: every selected logit is within the threshold of the true k-th logit
    kth = -np.sort(-R.logits, axis=1)[:, k - 1]
    sel = np.take_along_axis(R.logits, idx_gpu.astype(np.int64), 1)
    assert np.all(sel >= kth[:, None] - TIE_GAP), "selected an expert far below the k-th logit"
    assert np.all(np.sort(idx_gpu, 1)[:, 1:] != np.sort(idx_gpu, 1)[:, :-1]) if k > 1 else True
    same = np.all(idx_gpu == R.idx, axis=1)
    check_gates(gates_gpu[same], R.gates[same])
    return same
