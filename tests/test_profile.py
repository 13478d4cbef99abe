"""The kernel profiler (GPU): event brackets count every launch of a layer step, and the tensor-core
GEMM kernels report the SM clock they ran at (in-kernel clock64 cycles over globaltimer ns)."""
import pytest
import torch

from cases import case
from harness import to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

GEMMS = {"gemm_gate_up_swiglu", "gemm_down", "gemm_bwd_dgrad_down", "gemm_bwd_recompute_swiglu", "gemm_wgrad",
         "gemm_dgrad_x", "gemm_router_dx", "router_dwr"}


def test_profile_counts_launches_and_gemm_clocks(moe):
    c, inp, _ = case("ragged_mixtral")
    mc = moe.config_from(c)
    buf = moe.Buffers.allocate(mc)
    T, d, E, G, f = c["T"], c["d"], c["E"], c["E"] + c["S"], c["f"]
    x, W_r = to_dev_bf16(inp["x"]), to_dev(inp["W_r"])
    Wg, Wu, Wd, dy = (to_dev_bf16(inp[n]) for n in ("W_gate", "W_up", "W_down", "dy"))
    y, dx = torch.empty(T, d, dtype=torch.bfloat16, device="cuda"), torch.empty(T, d, dtype=torch.bfloat16,
                                                                                     device="cuda")
    dW_r = torch.empty(d, E, dtype=torch.float32, device="cuda")
    dWg, dWu = torch.empty(G, f, d, dtype=torch.bfloat16, device="cuda"), torch.empty(G, f, d, dtype=torch.bfloat16,
                                                                                        device="cuda")
    dWd = torch.empty(G, d, f, dtype=torch.bfloat16, device="cuda")
    moe.moe_profile_enable(True)
    for _ in range(2):
        moe.moe_layer_fwd(mc, x, W_r, None, Wg, Wu, Wd, y, buf.saved, buf.ws)
        moe.moe_layer_bwd(mc, x, W_r, None, Wg, Wu, Wd, buf.saved, dy, dx, dW_r, None, dWg, dWu, dWd, buf.ws)
    prof = moe.moe_profile_read()
    mhz = moe.moe_profile_sm_clock()
    moe.moe_profile_enable(False)
    assert moe.moe_check_error(buf.ws) == 0
    ran = {n for n, (ms, launches) in prof.items() if launches}
    assert {"route_fwd", "dispatch_gather", "combine", "router_dlogits", "combine_bwd"} <= ran
    assert all(prof[n][1] % 2 == 0 and prof[n][0] > 0 for n in ran)   # two steps, timed
    assert GEMMS <= ran
    # every GEMM that ran has a clock, nothing else does, and it is a clock an SM can run at
    assert set(mhz) == ran & GEMMS
    assert all(300.0 < v < 3000.0 for v in mhz.values()), mhz
    # disabled: the sums are cleared and nothing is recorded
    moe.moe_layer_fwd(mc, x, W_r, None, Wg, Wu, Wd, y, buf.saved, buf.ws)
    assert moe.moe_profile_sm_clock() == {}
