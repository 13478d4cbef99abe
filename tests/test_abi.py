"""The C-ABI library loads, exports every entry point include/moe.h declares, and its host-side
argument checks answer without a GPU (CPU only: no compute call is made)."""
import ctypes
import os
import re

import pytest

import mixture_experts_layer_10_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"^(?:moe_status_t|const char\*)\s+(moe_\w+)\s*\(", text, re.M)))


@pytest.fixture(scope="module")
def lib():
    return moe.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), f"libmoe.so does not export {n}"
    assert sorted(moe.EXPORTS) == names, "binding and header disagree"


def test_status_strings(lib):
    for code in range(7):
        assert moe.moe_status_string(code)
    assert moe.moe_status_string(3) == "workspace too small"


def test_workspace_size_and_rows():
    c = moe.config(T=8192, d=4096, f=14336, E=8, k=2)
    ws, saved = moe.moe_workspace_size(c)
    assert saved == 8192 * 2 * 8 + 8192 * 8 * 4          # idx, gates; the logits (256-aligned here)
    assert moe.moe_saved_layout(c) == (8192 * 2 * 8, 8192 * 8 * 4, saved, 0)
    rows = moe.moe_perm_rows(c)
    # routed rows padded per expert to 256, all segment starts multiples of 256
    assert rows % 256 == 0 and rows >= 8192 * 2 + 255 * 8
    assert ws > 3 * rows * 14336 * 2
    c2 = moe.config(T=16384, d=2048, f=1408, E=64, k=6, S=2, renorm=1)
    assert moe.moe_perm_rows(c2) >= 16384 * 6 + 2 * 16384
    # renormalised gates keep no logits; odd sizes start the logits and kept rows on 256 bytes
    assert moe.moe_saved_layout(c2)[:2] == (0, 0) and moe.moe_workspace_size(c2)[1] == 16384 * 6 * 8
    c3 = moe.config(T=100, d=64, f=64, E=3, k=1, keep_rows=256)
    lo, lb, ko, kb = moe.moe_saved_layout(c3)
    assert (lo, lb) == (1024, 1200) and ko == 2304 and kb == 2 * 256 * 64 * 2
    assert moe.moe_workspace_size(c3)[1] == ko + kb


@pytest.mark.parametrize("bad", [
    dict(T=0, d=128, f=256, E=8, k=2), dict(T=16, d=100, f=256, E=8, k=2),
    dict(T=16, d=128, f=96, E=8, k=2), dict(T=16, d=128, f=256, E=8, k=9),
    dict(T=16, d=128, f=256, E=300, k=2), dict(T=16, d=128, f=256, E=8, k=2, S=9),
    dict(T=16, d=128, f=256, E=8, k=0), dict(T=16, d=128, f=256, E=8, k=2, keep_rows=-1),
    dict(T=16, d=128, f=256, E=8, k=2, gather_in_gemm=2), dict(T=16, d=128, f=256, E=8, k=2, gather_in_gemm=-1),
])
def test_invalid_config_rejected(lib, bad):
    c = moe.config(**bad)
    ws, saved = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(c), ctypes.byref(ws), ctypes.byref(saved)) == 1


def test_null_and_misaligned_pointers_rejected(lib):
    c = moe.config(T=64, d=128, f=256, E=8, k=2)
    s = None
    # null x
    assert lib.moe_route(ctypes.byref(c), None, 0x10000, None, 0x20000, 0x30000, None, 0x40000, 1 << 30, s) == 1
    # misaligned W_r
    assert lib.moe_route(ctypes.byref(c), 0x10000, 0x20004, None, 0x30000, 0x40000, None, 0x50000, 1 << 30, s) == 1
    # workspace pointer must be 256-byte aligned
    assert lib.moe_combine(ctypes.byref(c), 0x10000, 0x20000, 0x30000, 0x40010, 1 << 30, s) == 1


def test_small_workspace_rejected(lib):
    c = moe.config(T=64, d=128, f=256, E=8, k=2)
    ws, _ = moe.moe_workspace_size(c)
    assert lib.moe_combine(ctypes.byref(c), 0x10000, 0x20000, 0x30000, 0x100000, ws - 1, None) == 3
    assert lib.moe_dispatch(ctypes.byref(c), 0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000,
                            0x70000, 0x100000, 16, None) == 3


def test_fp8_arguments_rejected(lib):
    # the quantiser: cols a multiple of 16, at most 16384; aligned pointers
    assert lib.moe_quantize_rows_e4m3(0x10000, 4, 16400, 0x20000, 0x30000, None) == 1
    assert lib.moe_quantize_rows_e4m3(0x10000, 4, 40, 0x20000, 0x30000, None) == 1
    assert lib.moe_quantize_rows_e4m3(0x10000, 4, 64, 0x20008, 0x30000, None) == 1
    assert lib.moe_quantize_rows_e4m3(0x10000, -1, 64, 0x20000, 0x30000, None) == 1
    c = moe.config(T=64, d=128, f=256, E=8, k=2)
    ws, _ = moe.moe_workspace_size(c)
    # null scale, misaligned codes
    assert lib.moe_down_fp8(ctypes.byref(c), 0x10000, None, 0x20000, 0x30000, 0x40000, 0x100000, ws, None) == 1
    assert lib.moe_gate_up_fp8(ctypes.byref(c), 0x10004, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000, 0x70000,
                               0x100000, ws, None) == 1
    assert lib.moe_layer_fwd_fp8(ctypes.byref(c), 0x10000, 0x20000, None, 0x30000, 0x40000, 0x50000, None,
                                 0x70000, 0x80000, 0x90000, 0xA0000, 0x100000, ws, None) == 1
    # kept activations cannot survive the FP8 forward's scratch
    ck = moe.config(T=64, d=128, f=256, E=8, k=2, keep_rows=256)
    wsk, _ = moe.moe_workspace_size(ck)
    assert lib.moe_layer_fwd_fp8(ctypes.byref(ck), 0x10000, 0x20000, None, 0x30000, 0x40000, 0x50000, 0x60000,
                                 0x70000, 0x80000, 0x90000, 0xA0000, 0x100000, wsk, None) == 1


def test_fp8_backward_arguments_rejected(lib):
    # the column quantiser: rows (top + bottom) a multiple of 16, a bottom exactly when it has rows
    assert lib.moe_quantize_cols_e4m3(0x10000, None, 2, 40, 0, 64, 0x20000, 0x30000, None) == 1
    assert lib.moe_quantize_cols_e4m3(0x10000, None, 2, 64, 64, 64, 0x20000, 0x30000, None) == 1
    assert lib.moe_quantize_cols_e4m3(0x10000, 0x18000, 2, 64, 0, 64, 0x20000, 0x30000, None) == 1
    assert lib.moe_quantize_cols_e4m3(0x10000, None, 2, 16384, 16400, 64, 0x20000, 0x30000, None) == 1
    assert lib.moe_quantize_cols_e4m3(0x10008, None, 2, 64, 0, 64, 0x20000, 0x30000, None) == 1
    c = moe.config(T=64, d=128, f=256, E=8, k=2)
    ws, _ = moe.moe_workspace_size(c)
    p = [0x10000 * (i + 1) for i in range(19)]
    # a null scale
    q = list(p)
    q[4] = None
    assert lib.moe_layer_bwd_fp8(ctypes.byref(c), *q, 0x1000000, ws, None) == 1
    # every row's a, b come from the codes: no kept activations
    ck = moe.config(T=64, d=128, f=256, E=8, k=2, keep_rows=256)
    wsk, _ = moe.moe_workspace_size(ck)
    assert lib.moe_layer_bwd_fp8(ctypes.byref(ck), *p, 0x1000000, wsk, None) == 1


def test_a_library_that_does_not_load_raises(tmp_path, monkeypatch):
    # no fallback: a broken library file is an error, never a silent CPU path
    bad = tmp_path / "libmoe.so"
    bad.write_bytes(b"not a shared object")
    monkeypatch.setattr(moe, "_lib", None)
    with pytest.raises(OSError):
        moe.load(str(bad))


def test_saved_layout_and_clock_query_arguments(lib):
    """The saved-layout query takes nullable outputs and rejects a bad configuration; the in-kernel
    clock query rejects a kernel id out of range or a missing output before touching a device."""
    c = moe.config(T=64, d=128, f=128, E=8, k=2)
    assert lib.moe_saved_layout(ctypes.byref(c), None, None, None, None) == 0
    bad = moe.config(T=16, d=100, f=256, E=8, k=2)
    out = ctypes.c_size_t()
    assert lib.moe_saved_layout(ctypes.byref(bad), ctypes.byref(out), None, None, None) == 1
    mhz = ctypes.c_double()
    n = len(moe.moe_profile_read())
    assert lib.moe_profile_sm_clock(-1, ctypes.byref(mhz)) == 1
    assert lib.moe_profile_sm_clock(n, ctypes.byref(mhz)) == 1
    assert lib.moe_profile_sm_clock(0, None) == 1
