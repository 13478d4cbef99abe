"""Python binding of the GB300 MoE FFN layer's C ABI (include/moe.h).

Argument marshalling only: every function below hands pointers and sizes to ``libmoe.so`` and
every step of the layer runs in its CUDA kernels.  PyTorch is used for device memory and streams.
There is no fallback: if the library is missing or fails to load, ``load()`` raises.

Tensors are passed as torch tensors (their ``data_ptr()``), ``None`` for optional ones.  bf16
tensors may be ``torch.bfloat16`` or any 16-bit dtype holding bf16 bits.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_BAD_INDEX", 6: "MOE_ERR_TIMEOUT"}

# Every entry point declared in include/moe.h.
EXPORTS = ("moe_workspace_size", "moe_perm_rows", "moe_workspace_init", "moe_route", "moe_dispatch",
           "moe_dispatch_noalloc",
           "moe_expert_ffn_fwd", "moe_combine", "moe_expert_ffn_bwd", "moe_router_bwd",
           "moe_combine_bwd", "moe_layer_fwd", "moe_layer_bwd", "moe_check_error",
           "moe_debug_inject", "moe_profile_enable", "moe_profile_read", "moe_status_string",
           "moe_quantize_rows_e4m3", "moe_gate_up_fp8", "moe_down_fp8", "moe_layer_fwd_fp8",
           "moe_keep_rows_for_budget", "moe_keep_rows_for_free_memory", "moe_quantize_cols_e4m3",
           "moe_layer_bwd_fp8", "moe_saved_layout", "moe_profile_sm_clock")


class moe_config_t(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("renorm", ctypes.c_int32), ("capacity_factor", ctypes.c_float),
                ("keep_rows", ctypes.c_int32), ("gather_in_gemm", ctypes.c_int32)]


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


_lib = None
_P = ctypes.c_void_p


def load(path: str | None = None):
    """Load libmoe.so (building it first if it is missing and nvcc is available)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        from . import _build
        _build.build()
    lib = ctypes.CDLL(path)
    cfgp = ctypes.POINTER(moe_config_t)
    sig = {
        "moe_workspace_size": [cfgp, ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)],
        "moe_perm_rows": [cfgp, ctypes.POINTER(ctypes.c_int64)],
        "moe_saved_layout": [cfgp] + [ctypes.POINTER(ctypes.c_size_t)] * 4,
        "moe_keep_rows_for_budget": [cfgp, ctypes.c_uint64, ctypes.POINTER(ctypes.c_int32),
                                     ctypes.POINTER(ctypes.c_uint64)],
        "moe_keep_rows_for_free_memory": [cfgp, ctypes.c_uint64, ctypes.POINTER(ctypes.c_int32),
                                          ctypes.POINTER(ctypes.c_uint64)],
        "moe_workspace_init": [cfgp, _P, ctypes.c_size_t, _P],
        "moe_route": [cfgp, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
        "moe_dispatch": [cfgp, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
        "moe_dispatch_noalloc": [cfgp, _P, _P, _P, _P, _P, _P, _P, _P, _P],
        "moe_expert_ffn_fwd": [cfgp, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
        "moe_combine": [cfgp, _P, _P, _P, _P, ctypes.c_size_t, _P],
        "moe_expert_ffn_bwd": [cfgp, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
        "moe_router_bwd": [cfgp, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
        "moe_combine_bwd": [cfgp, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
        "moe_quantize_rows_e4m3": [_P, ctypes.c_int64, ctypes.c_int32, _P, _P, _P],
        "moe_gate_up_fp8": [cfgp, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
        "moe_down_fp8": [cfgp, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
        "moe_layer_fwd_fp8": [cfgp, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
        "moe_quantize_cols_e4m3": [_P, _P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, _P,
                                   _P],
        "moe_layer_bwd_fp8": [cfgp] + [_P] * 20 + [ctypes.c_size_t, _P],
        "moe_layer_fwd": [cfgp, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
        "moe_layer_bwd": [cfgp, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                          ctypes.c_size_t, _P],
        "moe_check_error": [_P, _P],
        "moe_debug_inject": [_P, ctypes.c_int32, ctypes.c_int32, ctypes.c_uint64, _P],
        "moe_profile_enable": [ctypes.c_int32],
        "moe_profile_sm_clock": [ctypes.c_int32, ctypes.POINTER(ctypes.c_double)],
        "moe_profile_read": [ctypes.c_int32, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_double),
                             ctypes.POINTER(ctypes.c_int32)],
        "moe_status_string": [ctypes.c_int],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name == "moe_status_string" else ctypes.c_int
    _lib = lib
    return lib


# ------------------------------------------------------------------------------------------------
# marshalling helpers
# ------------------------------------------------------------------------------------------------

def config(T: int, d: int, f: int, E: int, k: int, S: int = 0, renorm: int = 0, cf: float = 0.0,
           keep_rows: int = 0, gather_in_gemm: int = 0):
    return moe_config_t(int(T), int(d), int(f), int(E), int(k), int(S), int(renorm), float(cf), int(keep_rows),
                        int(gather_in_gemm))


def config_from(c: dict) -> moe_config_t:
    """From a workload dict with keys T, d, f, E, k, S, renorm, cf (and keep_rows, gather_in_gemm,
    default 0)."""
    return config(c["T"], c["d"], c["f"], c["E"], c["k"], c.get("S", 0), c.get("renorm", 0), c.get("cf", 0.0),
                  c.get("keep_rows", 0), c.get("gather_in_gemm", 0))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, where: str):
    if code != MOE_OK:
        raise MoEError(code, where)


def _call(name, *args):
    _check(getattr(load(), name)(*args), name)


# ------------------------------------------------------------------------------------------------
# the C entry points, one to one
# ------------------------------------------------------------------------------------------------

def moe_workspace_size(cfg: moe_config_t):
    ws, saved = ctypes.c_size_t(), ctypes.c_size_t()
    _call("moe_workspace_size", ctypes.byref(cfg), ctypes.byref(ws), ctypes.byref(saved))
    return ws.value, saved.value


def moe_saved_layout(cfg: moe_config_t):
    """(logits_off, logits_bytes, kept_off, kept_bytes) of the `saved` buffer."""
    v = [ctypes.c_size_t() for _ in range(4)]
    _call("moe_saved_layout", ctypes.byref(cfg), *(ctypes.byref(x) for x in v))
    return tuple(x.value for x in v)


def moe_perm_rows(cfg: moe_config_t) -> int:
    r = ctypes.c_int64()
    _call("moe_perm_rows", ctypes.byref(cfg), ctypes.byref(r))
    return r.value


def moe_keep_rows_for_budget(cfg: moe_config_t, budget_bytes: int):
    """(keep_rows, kept bytes) for a byte budget of kept activations."""
    r, b = ctypes.c_int32(), ctypes.c_uint64()
    _call("moe_keep_rows_for_budget", ctypes.byref(cfg), int(budget_bytes), ctypes.byref(r), ctypes.byref(b))
    return r.value, b.value


def moe_keep_rows_for_free_memory(cfg: moe_config_t, reserve_bytes: int):
    """(keep_rows, kept bytes) for the current device's free memory less ``reserve_bytes``."""
    r, b = ctypes.c_int32(), ctypes.c_uint64()
    _call("moe_keep_rows_for_free_memory", ctypes.byref(cfg), int(reserve_bytes), ctypes.byref(r),
          ctypes.byref(b))
    return r.value, b.value


def moe_workspace_init(cfg, ws, stream=None):
    _call("moe_workspace_init", ctypes.byref(cfg), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


def moe_route(cfg, x, W_r, b_r, idx, gates, logits, ws, stream=None):
    _call("moe_route", ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(b_r), _ptr(idx), _ptr(gates),
          _ptr(logits), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


def moe_dispatch(cfg, idx, x, counts, offsets, row_of_slot, token_of_row, x_perm, ws, stream=None):
    _call("moe_dispatch", ctypes.byref(cfg), _ptr(idx), _ptr(x), _ptr(counts), _ptr(offsets),
          _ptr(row_of_slot), _ptr(token_of_row), _ptr(x_perm), _ptr(ws), ws.numel(), _stream(stream))


def moe_dispatch_noalloc(cfg, idx, x, counts, offsets, row_of_slot, token_of_row, x_perm, status=None,
                         stream=None):
    """moe_dispatch without a workspace (scratch in a fixed array inside the library); ``status``
    (optional int32 device tensor of one element) receives the call's device-side status."""
    _call("moe_dispatch_noalloc", ctypes.byref(cfg), _ptr(idx), _ptr(x), _ptr(counts), _ptr(offsets),
          _ptr(row_of_slot), _ptr(token_of_row), _ptr(x_perm), _ptr(status), _stream(stream))


def moe_expert_ffn_fwd(cfg, x_perm, W_gate, W_up, W_down, o_perm, ws, stream=None):
    _call("moe_expert_ffn_fwd", ctypes.byref(cfg), _ptr(x_perm), _ptr(W_gate), _ptr(W_up), _ptr(W_down),
          _ptr(o_perm), _ptr(ws), ws.numel(), _stream(stream))


def moe_combine(cfg, o_perm, gates, y, ws, stream=None):
    _call("moe_combine", ctypes.byref(cfg), _ptr(o_perm), _ptr(gates), _ptr(y), _ptr(ws), ws.numel(),
          _stream(stream))


def moe_expert_ffn_bwd(cfg, x_perm, dy, gates, W_gate, W_up, W_down, dx_perm, dgates,
                       dW_gate, dW_up, dW_down, ws, stream=None):
    _call("moe_expert_ffn_bwd", ctypes.byref(cfg), _ptr(x_perm), _ptr(dy), _ptr(gates), _ptr(W_gate),
          _ptr(W_up), _ptr(W_down), _ptr(dx_perm), _ptr(dgates), _ptr(dW_gate), _ptr(dW_up),
          _ptr(dW_down), _ptr(ws), ws.numel(), _stream(stream))


def moe_router_bwd(cfg, x, W_r, b_r, idx, gates, dgates, dlogits, dW_r, db_r, ws, stream=None):
    _call("moe_router_bwd", ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(b_r), _ptr(idx), _ptr(gates),
          _ptr(dgates), _ptr(dlogits), _ptr(dW_r), _ptr(db_r), _ptr(ws), ws.numel(), _stream(stream))


def moe_combine_bwd(cfg, dx_perm, dlogits, W_r, dx, ws, stream=None):
    _call("moe_combine_bwd", ctypes.byref(cfg), _ptr(dx_perm), _ptr(dlogits), _ptr(W_r), _ptr(dx),
          _ptr(ws), ws.numel(), _stream(stream))


def moe_quantize_rows_e4m3(src, codes, scales, stream=None):
    """src [rows, cols] bf16 -> codes [rows, cols] uint8, scales [rows] fp32."""
    rows, cols = src.shape[0], src.shape[-1]
    _call("moe_quantize_rows_e4m3", _ptr(src), int(src.numel() // cols) if rows else 0, int(cols), _ptr(codes),
          _ptr(scales), _stream(stream))


def moe_gate_up_fp8(cfg, x8, x_scale, wg8, wg_scale, wu8, wu_scale, h, ws, stream=None):
    _call("moe_gate_up_fp8", ctypes.byref(cfg), _ptr(x8), _ptr(x_scale), _ptr(wg8), _ptr(wg_scale), _ptr(wu8),
          _ptr(wu_scale), _ptr(h), _ptr(ws), ws.numel(), _stream(stream))


def moe_down_fp8(cfg, h8, h_scale, wd8, wd_scale, o_perm, ws, stream=None):
    _call("moe_down_fp8", ctypes.byref(cfg), _ptr(h8), _ptr(h_scale), _ptr(wd8), _ptr(wd_scale), _ptr(o_perm),
          _ptr(ws), ws.numel(), _stream(stream))


def moe_layer_fwd_fp8(cfg, x, W_r, b_r, wg8, wg_scale, wu8, wu_scale, wd8, wd_scale, y, saved, ws, stream=None):
    _call("moe_layer_fwd_fp8", ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(b_r), _ptr(wg8), _ptr(wg_scale),
          _ptr(wu8), _ptr(wu_scale), _ptr(wd8), _ptr(wd_scale), _ptr(y), _ptr(saved), _ptr(ws), ws.numel(),
          _stream(stream))


def moe_quantize_cols_e4m3(top, bottom, codes, scales, stream=None):
    """top [G, r1, cols] (and bottom [G, r2, cols] or None) bf16 -> codes [G, cols, r1 + r2] uint8 and
    scales [G, cols] fp32: per-column codes of the stacked source, transposed."""
    G, r1, cols = top.shape
    r2 = 0 if bottom is None else bottom.shape[1]
    _call("moe_quantize_cols_e4m3", _ptr(top), _ptr(bottom), int(G), int(r1), int(r2), int(cols), _ptr(codes),
          _ptr(scales), _stream(stream))


def moe_layer_bwd_fp8(cfg, x, W_r, b_r, wg8, wg_scale, wu8, wu_scale, wdt8, wdt_scale, wgut8, wgut_scale, saved, dy,
                      dx, dW_r, db_r, dW_gate, dW_up, dW_down, ws, stream=None):
    _call("moe_layer_bwd_fp8", ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(b_r), _ptr(wg8), _ptr(wg_scale),
          _ptr(wu8), _ptr(wu_scale), _ptr(wdt8), _ptr(wdt_scale), _ptr(wgut8), _ptr(wgut_scale), _ptr(saved),
          _ptr(dy), _ptr(dx), _ptr(dW_r), _ptr(db_r), _ptr(dW_gate), _ptr(dW_up), _ptr(dW_down), _ptr(ws),
          ws.numel(), _stream(stream))


def moe_layer_fwd(cfg, x, W_r, b_r, W_gate, W_up, W_down, y, saved, ws, stream=None):
    _call("moe_layer_fwd", ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(b_r), _ptr(W_gate), _ptr(W_up),
          _ptr(W_down), _ptr(y), _ptr(saved), _ptr(ws), ws.numel(), _stream(stream))


def moe_layer_bwd(cfg, x, W_r, b_r, W_gate, W_up, W_down, saved, dy, dx, dW_r, db_r,
                  dW_gate, dW_up, dW_down, ws, stream=None):
    _call("moe_layer_bwd", ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(b_r), _ptr(W_gate), _ptr(W_up),
          _ptr(W_down), _ptr(saved), _ptr(dy), _ptr(dx), _ptr(dW_r), _ptr(db_r), _ptr(dW_gate),
          _ptr(dW_up), _ptr(dW_down), _ptr(ws), ws.numel(), _stream(stream))


def moe_check_error(ws, stream=None) -> int:
    """Synchronise and return (and clear) the first device-side status recorded in ws."""
    return load().moe_check_error(_ptr(ws), _stream(stream))


def moe_debug_inject(ws, stall_block: int, timeout_ns: int, stream=None, stall_fill: int = -1):
    _call("moe_debug_inject", _ptr(ws), int(stall_block), int(stall_fill), int(timeout_ns), _stream(stream))


def moe_profile_enable(on: bool):
    _call("moe_profile_enable", int(bool(on)))


def moe_profile_read() -> dict:
    """{kernel name: (total ms, launches)} for every kernel of the library (waits for the events)."""
    out, i = {}, 0
    name, ms, n = ctypes.c_char_p(), ctypes.c_double(), ctypes.c_int32()
    while True:
        code = load().moe_profile_read(i, ctypes.byref(name), ctypes.byref(ms), ctypes.byref(n))
        if code == 1:
            return out
        _check(code, "moe_profile_read")
        out[name.value.decode()] = (ms.value, n.value)
        i += 1


def moe_profile_sm_clock() -> dict:
    """{kernel name: mean SM MHz} of the tensor-core GEMM kernels that ran since
    moe_profile_enable (in-kernel clock64 over globaltimer; synchronises the device)."""
    names = moe_profile_read()
    out = {}
    mhz = ctypes.c_double()
    for i, name in enumerate(names):
        _call("moe_profile_sm_clock", i, ctypes.byref(mhz))
        if mhz.value > 0:
            out[name] = mhz.value
    return out


def moe_status_string(code: int) -> str:
    return load().moe_status_string(int(code)).decode()


# ------------------------------------------------------------------------------------------------
# buffers of one layer instance
# ------------------------------------------------------------------------------------------------

@dataclass
class Buffers:
    """Device buffers a layer instance needs: the workspace (header initialised) and `saved`."""
    cfg: moe_config_t
    ws: object
    saved: object
    rows: int

    @classmethod
    def allocate(cls, cfg: moe_config_t, device="cuda", stream=None):
        import torch
        ws_bytes, saved_bytes = moe_workspace_size(cfg)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
        saved = torch.empty(saved_bytes, dtype=torch.uint8, device=device)
        moe_workspace_init(cfg, ws, stream)
        return cls(cfg, ws, saved, moe_perm_rows(cfg))

    def saved_views(self):
        """Views of `saved`: idx int32 [T,k], gates fp32 [T,k], logits fp32 [T,E] (None with
        renormalised gates, which keep none)."""
        import torch
        T, k, E = self.cfg.T, self.cfg.k, self.cfg.E
        idx = self.saved[:4 * T * k].view(torch.int32).view(T, k)
        gates = self.saved[4 * T * k:8 * T * k].view(torch.float32).view(T, k)
        off, nbytes, _, _ = moe_saved_layout(self.cfg)
        logits = self.saved[off:off + nbytes].view(torch.float32).view(T, E) if nbytes else None
        return idx, gates, logits
