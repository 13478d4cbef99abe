"""moe_dispatch_noalloc, the dispatch for callers that cannot allocate device memory (GPU).

Such callers (code inside a framework-owned memory arena, or on a path where cudaMalloc and its
implicit synchronisation are not allowed) get no workspace argument; the entry point keeps its
scratch in a fixed array inside the library.  This file checks, through the C ABI, that two calls
in a row each give exactly what moe_dispatch (with its own workspace) gives on the same inputs --
the second call must not see anything the first one left in the shared array -- and that sizes
beyond the array's limit are refused without work.  It is collected last so that a failure here
leaves every other test already run; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _outputs(T, k, E, rows, d):
    return dict(counts=torch.full((E,), -1, dtype=torch.int32, device="cuda"),
                offsets=torch.full((E + 1,), -1, dtype=torch.int32, device="cuda"),
                row_of_slot=torch.full((T * k,), -9, dtype=torch.int32, device="cuda"),
                token_of_row=torch.full((T * k,), -9, dtype=torch.int32, device="cuda"),
                x_perm=torch.zeros(rows, d, dtype=torch.bfloat16, device="cuda"))


def _same(a, b):
    for key in a:
        assert torch.equal(a[key].view(torch.int16) if a[key].dtype == torch.bfloat16 else a[key],
                           b[key].view(torch.int16) if b[key].dtype == torch.bfloat16 else b[key]), key


@pytest.mark.parametrize("T,d,E,k,S,cf,skew", [(3000, 256, 16, 4, 1, 0.0, 0.0), (2000, 128, 8, 2, 0, 1.0, 1.5)])
def test_no_alloc_dispatch_matches_workspace_dispatch(moe, T, d, E, k, S, cf, skew):
    mc = moe.config(T=T, d=d, f=64, E=E, k=k, S=S, cf=cf)
    buf = moe.Buffers.allocate(mc)
    rows = buf.rows
    for call, seed in enumerate((21, 22)):                    # two calls in a row
        idx = torch.from_numpy(synth.random_assignments(seed, T, E, k, skew)).cuda()
        x = torch.from_numpy(synth.normal_bf16(seed, "x", (T, d), 1.0).view(np.int16)).view(torch.bfloat16).cuda()
        ref = _outputs(T, k, E, rows, d)
        moe.moe_dispatch(mc, idx, x, ref["counts"], ref["offsets"], ref["row_of_slot"], ref["token_of_row"],
                         ref["x_perm"], buf.ws)
        assert moe.moe_check_error(buf.ws) == 0
        got = _outputs(T, k, E, rows, d)
        moe.moe_dispatch_noalloc(mc, idx, x, got["counts"], got["offsets"], got["row_of_slot"],
                                 got["token_of_row"], got["x_perm"])
        torch.cuda.synchronize()
        _same(got, ref)
        assert int(got["counts"].sum()) == T * k, f"call {call}"


def test_no_alloc_dispatch_refuses_sizes_beyond_its_scratch(moe):
    T, k, E, d = 70000, 4, 16, 64                             # 280000 assignments > 262144
    mc = moe.config(T=T, d=d, f=64, E=E, k=k)
    t = torch.empty(16, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoEError) as e:
        moe.moe_dispatch_noalloc(mc, t, t, t, t, t, t, t)
    assert e.value.code == 2
