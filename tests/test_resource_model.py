"""The analytical resource model against the library's own sizes and the closed-form FLOP counts
(CPU: the library is loaded but runs nothing on a GPU)."""
import pytest

import mixture_experts_layer_10_gb300 as moe
from mixture_experts_layer_10_gb300 import resource_model as rm
import synth

WORKLOADS = ["tiny", "mixtral", "deepseek", "qwen3", "gptoss"]


@pytest.mark.parametrize("name", WORKLOADS)
def test_rows_and_workspace_match_the_library(name):
    cfg = synth.CONFIGS[name]
    mc = moe.config_from(cfg)
    ws, saved = moe.moe_workspace_size(mc)
    mem = rm.memory(cfg)
    assert mem["padded_rows"] == moe.moe_perm_rows(mc)
    assert mem["saved"] == saved
    # the model leaves out headers, tables and alignment: within 1% of the library's figure
    assert abs(mem["workspace"] - ws) <= 0.01 * ws, (mem["workspace"], ws)


@pytest.mark.parametrize("name", WORKLOADS)
def test_gemm_flops_closed_form(name):
    cfg = synth.CONFIGS[name]
    T, d, f, k, S = cfg["T"], cfg["d"], cfg["f"], cfg["k"], cfg["S"]
    R = T * k + S * T
    assert rm.gemm_flops(cfg) == 22 * R * d * f            # with recompute
    assert rm.gemm_flops(cfg, kept_rows=R) == 18 * R * d * f   # every row's a, b kept


def test_kept_activation_bytes():
    cfg = dict(synth.CONFIGS["mixtral"], keep_rows=1000)
    assert rm.memory(cfg)["kept_activations"] == 768 * 14336 * 4    # rounded down to 256 rows
    # the fused calls keep them in `saved`, after idx, gates and the logits (each from a 256-byte
    # boundary)
    _, saved = moe.moe_workspace_size(moe.config_from(cfg))
    assert saved == rm.memory(cfg)["saved"] == 8192 * 2 * 8 + 8192 * 8 * 4 + 768 * 14336 * 4


@pytest.mark.parametrize("name", WORKLOADS)
def test_keep_rows_for_budget(name):
    """The library's budget rule: whole 256-row tiles of 4 d_ff bytes each, as many as fit, at
    most every row; `saved` then grows by exactly the kept bytes."""
    cfg = synth.CONFIGS[name]
    mc = moe.config_from(cfg)
    cap = moe.moe_perm_rows(mc)
    per_tile = 256 * 4 * cfg["f"]
    _, saved0 = moe.moe_workspace_size(mc)
    for budget in [0, per_tile - 1, per_tile, 3 * per_tile + 17, 10 ** 9, 1 << 62]:
        rows, kept = moe.moe_keep_rows_for_budget(mc, budget)
        assert rows == rm.keep_rows_for_budget(cfg, budget)
        assert rows % 256 == 0 and 0 <= rows <= cap
        assert kept == rows * 4 * cfg["f"] <= budget
        assert rows == cap or kept + per_tile > budget          # one more tile would not fit
        _, saved = moe.moe_workspace_size(moe.config_from(dict(cfg, keep_rows=rows)))
        assert saved - (saved0 + 255) // 256 * 256 == kept if rows else saved == saved0
    assert moe.moe_keep_rows_for_budget(mc, 1 << 62)[0] == cap


def test_router_columns():
    # stacked hi | mid | lo parts for narrow routers, three padded blocks up to 128 experts
    assert [rm.router_n(E, 2) for E in (1, 8, 9, 16, 24, 32, 64)] == [32, 32, 48, 48, 96, 96, 192]
    assert rm.router_n(33, 2) == 384 // 2
    assert rm.router_n(96, 8) == 384 and rm.router_n(128, 4) == 384 and rm.router_n(200, 4) == 200
    assert rm.router_n(24, 10) == 24


def test_prediction_is_a_roofline():
    cfg = synth.CONFIGS["mixtral"]
    p = rm.predict_ms(cfg, tensor_tflops=1000.0, hbm_gbs=5000.0)
    assert p["per_kernel_ms"]["gemm_wgrad"] == pytest.approx(rm.work(cfg)["gemm_wgrad"]["flops"] / 1e12)
    assert p["per_kernel_ms"]["combine"] == pytest.approx(rm.work(cfg)["combine"]["bytes"] / 5e9)
    assert p["step_ms"] > sum(v for v in p["per_kernel_ms"].values())


@pytest.mark.parametrize("name", WORKLOADS)
def test_forward_work_closed_forms(name):
    cfg = synth.CONFIGS[name]
    T, d, f, k, S = cfg["T"], cfg["d"], cfg["f"], cfg["k"], cfg["S"]
    R = T * k + S * T
    bf = rm.work_forward(cfg)
    q = rm.work_forward(cfg, fp8=True)
    # the same 6 R d f GEMM FLOPs, in bf16 or in e4m3
    assert sum(v["flops"] for n, v in bf.items() if n.startswith("gemm_")) == 6 * R * d * f
    assert sum(v.get("fp8_flops", 0) for v in q.values()) == 6 * R * d * f
    # the FP8 forward gathers one-byte codes: half the rows' bytes of the bf16 gather, plus scales
    meta = 12 * T * k
    assert q["dispatch_gather"]["bytes"] - 8 * R - meta == (bf["dispatch_gather"]["bytes"] - meta) // 2
    # its quantisation passes read bf16 and write codes once: x over T rows, h over R rows
    assert q["quantize_e4m3 (x)"]["bytes"] == 3 * T * d + 4 * T
    assert q["quantize_e4m3 (h)"]["bytes"] == 3 * R * f + 4 * R


def test_forward_prediction_runs_fp8_at_twice_the_rate():
    cfg = synth.CONFIGS["mixtral"]
    bf = rm.predict_forward_ms(cfg, tensor_tflops=1000.0, hbm_gbs=5000.0)
    q = rm.predict_forward_ms(cfg, tensor_tflops=1000.0, hbm_gbs=5000.0, fp8=True)
    assert q["per_kernel_ms"]["gemm_gate_up_fp8"] == pytest.approx(bf["per_kernel_ms"]["gemm_gate_up_swiglu"] / 2)
    assert q["per_kernel_ms"]["gemm_down_fp8"] == pytest.approx(bf["per_kernel_ms"]["gemm_down"] / 2)
    assert q["step_ms"] < bf["step_ms"]


def test_kernel_source_hash_ignores_comments_only():
    import bench
    a = "int f(int x) {  // doubles\n  return 2 * x; /* twice */ }\n"
    b = "int f(int x) {\n  /* a different\n comment */ return 2 * x; }"
    assert bench.code_only(a) == bench.code_only(b) == "int f(int x) { return 2 * x; }"
    assert bench.code_only(a) != bench.code_only(a.replace("2 *", "3 *"))


def test_padded_routed_rows():
    assert rm.padded_routed_rows([0, 1, 256, 257, 512]) == 0 + 256 + 256 + 512 + 512
    assert rm.padded_routed_rows([]) == 0


@pytest.mark.parametrize("name", WORKLOADS)
def test_calibrated_model_is_above_the_roofline(name):
    """The calibrated prediction adds padded rows, efficiencies below 1 and fixed costs to the same
    work: never faster than the roofline, and its GEMM share is the roofline's over EFF_GEMM (equal
    loads, rows a multiple of the tile)."""
    cfg = synth.CONFIGS[name]
    r = rm.predict_ms(cfg, tensor_tflops=1800.0, hbm_gbs=6800.0)
    c = rm.predict_ms_calibrated(cfg, tensor_tflops=1800.0, hbm_gbs=6800.0)
    assert c["step_ms"] > r["step_ms"]
    for n, t in r["per_kernel_ms"].items():
        if n.startswith("gemm_") and n != "gemm_router_dx":
            assert c["per_kernel_ms"][n] >= t / rm.EFF_GEMM * (1 - 1e-12)


def test_calibrated_model_charges_padding():
    cfg = synth.CONFIGS["qwen3"]
    N = cfg["T"] * cfg["k"]
    even = rm.predict_ms_calibrated(cfg, 1800.0, 6800.0)
    skew = [N - 127 * 10] + [10] * 127            # one large expert, 127 with 10 rows each
    c = rm.predict_ms_calibrated(cfg, 1800.0, 6800.0, counts=skew)
    assert c["padded_rows"] == rm.padded_routed_rows(skew)
    assert c["per_kernel_ms"]["gemm_wgrad"] > even["per_kernel_ms"]["gemm_wgrad"]
