"""Device-side error reporting without faulting the GPU (GPU).

* An expert id outside [0, E) comes back as MOE_ERR_BAD_INDEX through moe_check_error and empties
  that dispatch (no rows: offsets all 0, row_of_slot all -1); the next clean call succeeds.
* A bounded wait that runs out: the test hook makes one dispatch-scan block never publish its
  counts, the look-back of the blocks after it gives up after a short limit, the call reports
  MOE_ERR_TIMEOUT and downstream kernels see empty tables; the next clean call succeeds.
* The same in an expert GEMM: one operand stage never arrives, the MMA's wait gives up, the kernel
  drains what it has in flight, and the next call matches a call made before the stall.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import from_dev, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

BAD_INDEX, TIMEOUT = 5, 6


def _bufs(moe, T, d, E, k):
    mc = moe.config(T=T, d=d, f=64, E=E, k=k)
    buf = moe.Buffers.allocate(mc)
    out = dict(counts=torch.empty(E, dtype=torch.int32, device="cuda"),
               offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
               row_of_slot=torch.empty(T * k, dtype=torch.int32, device="cuda"),
               token_of_row=torch.empty(T * k, dtype=torch.int32, device="cuda"),
               x_perm=torch.zeros(buf.rows, d, dtype=torch.bfloat16, device="cuda"))
    return mc, buf, out


def _dispatch(moe, mc, buf, o, idx, x):
    moe.moe_dispatch(mc, idx, x, o["counts"], o["offsets"], o["row_of_slot"], o["token_of_row"],
                     o["x_perm"], buf.ws)


def test_bad_expert_index_is_reported(moe):
    T, d, E, k = 300, 64, 8, 2
    mc, buf, o = _bufs(moe, T, d, E, k)
    idx_np = synth.random_assignments(3, T, E, k)
    bad = idx_np.copy()
    bad[5, 1] = E
    bad[17, 0] = -3
    x = to_dev_bf16(synth.normal_bf16(3, "x", (T, d), 1.0))
    _dispatch(moe, mc, buf, o, to_dev(bad), x)
    assert moe.moe_check_error(buf.ws) == BAD_INDEX
    valid = bad[(bad >= 0) & (bad < E)]
    assert np.array_equal(from_dev(o["counts"]), np.bincount(valid, minlength=E))
    assert np.all(from_dev(o["offsets"]) == 0)
    assert np.all(from_dev(o["row_of_slot"]) == -1)
    # the error is cleared by the check; a clean call then matches the oracle
    _dispatch(moe, mc, buf, o, to_dev(idx_np), x)
    assert moe.moe_check_error(buf.ws) == 0
    D = oracle.dispatch(idx_np, E, None)
    assert np.array_equal(from_dev(o["counts"]), D.counts)
    assert np.array_equal(from_dev(o["row_of_slot"]).reshape(T, k), D.row_of_slot)


def test_stalled_scan_block_times_out(moe):
    T, d, E, k = 5000, 64, 16, 2          # 10000 assignments: three scan blocks
    mc, buf, o = _bufs(moe, T, d, E, k)
    idx_np = synth.random_assignments(4, T, E, k)
    x = to_dev_bf16(synth.normal_bf16(4, "x", (T, d), 1.0))
    moe.moe_debug_inject(buf.ws, 0, 20_000_000)      # block 0 never publishes; 20 ms limit
    _dispatch(moe, mc, buf, o, to_dev(idx_np), x)
    assert moe.moe_check_error(buf.ws) == TIMEOUT
    moe.moe_debug_inject(buf.ws, -1, 0)
    _dispatch(moe, mc, buf, o, to_dev(idx_np), x)
    assert moe.moe_check_error(buf.ws) == 0
    D = oracle.dispatch(idx_np, E, None)
    assert np.array_equal(from_dev(o["counts"]), D.counts)
    assert np.array_equal(from_dev(o["offsets"]), D.offsets)
    assert np.array_equal(from_dev(o["row_of_slot"]).reshape(T, k), D.row_of_slot)


def test_stalled_gemm_times_out_and_drains(moe):
    """An expert GEMM whose operand stage never arrives (the test hook makes the first CTA pair
    skip one fill): the MMA thread's bounded wait runs out and the call reports MOE_ERR_TIMEOUT.
    The kernel waits for the loads and MMAs it has in flight before it frees shared memory and
    TMEM, so the next call runs normally and gives bit for bit what a call before the stall gave."""
    from cases import case
    c, inp, L = case("ragged_mixtral")
    T, d, k, E = c["T"], c["d"], c["k"], c["E"]
    mc = moe.config_from(c)
    buf = moe.Buffers.allocate(mc)
    scratch = [torch.empty(n, dtype=torch.int32, device="cuda") for n in (E, E + 1, T * k, T * k)]
    x_perm = torch.empty(buf.rows, d, dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch(mc, to_dev(L.routing().idx.astype(np.int32)), to_dev_bf16(inp["x"]), *scratch, x_perm, buf.ws)
    Wg, Wu, Wd = (to_dev_bf16(inp[n]) for n in ("W_gate", "W_up", "W_down"))

    def ffn():
        o = torch.zeros(buf.rows, d, dtype=torch.bfloat16, device="cuda")
        moe.moe_expert_ffn_fwd(mc, x_perm, Wg, Wu, Wd, o, buf.ws)
        return o
    ref = ffn()
    assert moe.moe_check_error(buf.ws) == 0
    moe.moe_debug_inject(buf.ws, -1, 20_000_000, stall_fill=2)       # 20 ms bound
    ffn()
    assert moe.moe_check_error(buf.ws) == TIMEOUT
    moe.moe_debug_inject(buf.ws, -1, 0)
    again = ffn()
    assert moe.moe_check_error(buf.ws) == 0
    assert torch.equal(again.view(torch.int16), ref.view(torch.int16))


def test_invalid_arguments_enqueue_nothing(moe):
    mc = moe.config(T=64, d=128, f=128, E=4, k=2)
    buf = moe.Buffers.allocate(mc)
    y = torch.empty(64, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoEError) as e:
        moe.moe_combine(mc, None, None, y, buf.ws)
    assert e.value.code == 1
    small = buf.ws[: buf.ws.numel() // 2]
    with pytest.raises(moe.MoEError) as e:
        moe.moe_combine(mc, y, y, y, small)
    assert e.value.code == 3
    assert moe.moe_check_error(buf.ws) == 0
