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


def test_prediction_is_a_roofline():
    cfg = synth.CONFIGS["mixtral"]
    p = rm.predict_ms(cfg, tensor_tflops=1000.0, hbm_gbs=5000.0)
    assert p["per_kernel_ms"]["gemm_wgrad"] == pytest.approx(rm.work(cfg)["gemm_wgrad"]["flops"] / 1e12)
    assert p["per_kernel_ms"]["combine"] == pytest.approx(rm.work(cfg)["combine"]["bytes"] / 5e9)
    assert p["step_ms"] > sum(v for v in p["per_kernel_ms"].values())
