"""moe_dispatch_noalloc, the dispatch for callers that cannot allocate device memory (GPU).

Such callers (code inside a framework-owned memory arena, or on a path where cudaMalloc and its
implicit synchronisation are not allowed) get no workspace argument; the entry point keeps its
scratch in a fixed array inside the library.  This file checks, through the C ABI, on two calls in
a row:
  * each call gives exactly what moe_dispatch (with its own workspace) gives on the same inputs --
    the second call must not see anything the first one left in the shared array;
  * each call's counts, offsets, row_of_slot, token_of_row and x_perm equal the oracle's dispatch
    queues (the padded layout of include/moe.h, pad rows zero), and its status word reads MOE_OK;
  * an expert id out of range sets the status word to MOE_ERR_BAD_INDEX and empties the dispatch
    as documented, and the next clean call is correct again;
  * sizes beyond the array's limit are refused without work.
It is collected last so that a failure here leaves every other test already run; it also passes on
its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import from_dev, from_dev_bf16, padded_starts

pytestmark = pytest.mark.gpu

BAD_INDEX = 5


def _outputs(T, k, E, rows, d):
    return dict(counts=torch.full((E,), -1, dtype=torch.int32, device="cuda"),
                offsets=torch.full((E + 1,), -1, dtype=torch.int32, device="cuda"),
                row_of_slot=torch.full((T * k,), -9, dtype=torch.int32, device="cuda"),
                token_of_row=torch.full((T * k,), -9, dtype=torch.int32, device="cuda"),
                x_perm=torch.full((rows, d), 7.0, dtype=torch.bfloat16, device="cuda"))


def _same(a, b):
    for key in a:
        assert torch.equal(a[key].view(torch.int16) if a[key].dtype == torch.bfloat16 else a[key],
                           b[key].view(torch.int16) if b[key].dtype == torch.bfloat16 else b[key]), key


def _noalloc(moe, mc, idx, x, o):
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    moe.moe_dispatch_noalloc(mc, idx, x, o["counts"], o["offsets"], o["row_of_slot"], o["token_of_row"],
                             o["x_perm"], status)
    torch.cuda.synchronize()
    return int(status.item())


def _check_against_oracle(o, idx_np, x_bits, T, d, E, k, S, C):
    D = oracle.dispatch(idx_np, E, C)
    assert np.array_equal(from_dev(o["counts"]), D.counts)
    assert np.array_equal(from_dev(o["offsets"]), D.offsets)
    assert np.array_equal(from_dev(o["row_of_slot"]).reshape(T, k), D.row_of_slot)
    n = int(D.offsets[E])
    assert np.array_equal(from_dev(o["token_of_row"])[:n], D.token_of_row)
    # the padded expert-ordered rows: kept rows are copies of their token's x, pads are zero
    kept = np.concatenate([D.kept, np.full(S, T, dtype=np.int64)])
    P = padded_starts(kept)
    xp = from_dev_bf16(o["x_perm"])
    x = oracle.bf16_to_f64(x_bits)
    for g in range(E + S):
        toks = D.token_of_row[D.offsets[g]:D.offsets[g + 1]] if g < E else np.arange(T)
        assert np.array_equal(xp[P[g]:P[g] + kept[g]], x[toks]), f"segment {g}"
        assert np.all(xp[P[g] + kept[g]:P[g + 1]] == 0), f"pad rows of segment {g}"


@pytest.mark.parametrize("T,d,E,k,S,cf,skew", [(3000, 256, 16, 4, 1, 0.0, 0.0), (2000, 128, 8, 2, 0, 1.0, 1.5)])
def test_no_alloc_dispatch_matches_workspace_dispatch(moe, T, d, E, k, S, cf, skew):
    mc = moe.config(T=T, d=d, f=64, E=E, k=k, S=S, cf=cf)
    buf = moe.Buffers.allocate(mc)
    rows = buf.rows
    C = oracle.capacity_of(T, k, E, cf)
    for call, seed in enumerate((21, 22)):                    # two calls in a row
        idx_np = synth.random_assignments(seed, T, E, k, skew)
        x_bits = synth.normal_bf16(seed, "x", (T, d), 1.0)
        idx = torch.from_numpy(idx_np).cuda()
        x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda()
        ref = _outputs(T, k, E, rows, d)
        moe.moe_dispatch(mc, idx, x, ref["counts"], ref["offsets"], ref["row_of_slot"], ref["token_of_row"],
                         ref["x_perm"], buf.ws)
        assert moe.moe_check_error(buf.ws) == 0
        got = _outputs(T, k, E, rows, d)
        assert _noalloc(moe, mc, idx, x, got) == 0, f"call {call}: status"
        _same(got, ref)
        _check_against_oracle(got, idx_np, x_bits, T, d, E, k, S, C)


def test_no_alloc_dispatch_reports_a_bad_expert_id(moe):
    T, d, E, k, S = 1500, 128, 8, 2, 1
    mc = moe.config(T=T, d=d, f=64, E=E, k=k, S=S)
    rows = moe.moe_perm_rows(mc)
    idx_np = synth.random_assignments(31, T, E, k)
    x_bits = synth.normal_bf16(31, "x", (T, d), 1.0)
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda()
    bad = idx_np.copy()
    bad[700, 1] = E
    o = _outputs(T, k, E, rows, d)
    assert _noalloc(moe, mc, torch.from_numpy(bad).cuda(), x, o) == BAD_INDEX
    # documented outcome: the valid ids' demand, and no rows at all
    valid = bad[(bad >= 0) & (bad < E)]
    assert np.array_equal(from_dev(o["counts"]), np.bincount(valid, minlength=E))
    assert np.all(from_dev(o["offsets"]) == 0)
    assert np.all(from_dev(o["row_of_slot"]) == -1)
    assert np.all(from_dev(o["token_of_row"]) == -9)
    assert torch.all(o["x_perm"] == 7.0)
    # the next clean call starts afresh
    o = _outputs(T, k, E, rows, d)
    assert _noalloc(moe, mc, torch.from_numpy(idx_np).cuda(), x, o) == 0
    _check_against_oracle(o, idx_np, x_bits, T, d, E, k, S, None)


def test_no_alloc_dispatch_refuses_sizes_beyond_its_scratch(moe):
    T, k, E, d = 70000, 4, 16, 64                             # 280000 assignments > 262144
    mc = moe.config(T=T, d=d, f=64, E=E, k=k)
    t = torch.empty(16, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoEError) as e:
        moe.moe_dispatch_noalloc(mc, t, t, t, t, t, t, t, t)
    assert e.value.code == 2
