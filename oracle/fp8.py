"""FP8 (e4m3) quantisation step and the quantised gate/up projection, for the oracle.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only tests and bench.py's CPU leg use it.

The pages name mixed-precision / quantised experts only as a direction ("MoEBlaze" summary,
limitations and future work); they fix no format.  The plainest reading taken here:

* the format is OCP FP8 E4M3 (the "fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3
  mantissa bits; no infinities; the largest finite magnitude is 448 (exponent 15, mantissa 6);
  exponent field 0 holds the subnormals m * 2^-9; pattern S.1111.111 is NaN and never produced;
* a row of values v (bf16 widened exactly) is scaled by s = amax / 448 with amax = max |v| over
  the row, computed in fp32 (s = 1 when the row is all zero); each element is then v / s in fp32,
  rounded to the nearest e4m3 value with ties to the even mantissa, and saturated to +-448;
* an activation row and a weight row (one output channel) are quantised this way, so
  x . w ~= s_x s_w (q_x . q_w), exactly the fp64 product of the decoded codes and the scales.

Both rounding decisions (the fp32 division and the e4m3 rounding) are taken in fp32, as the
kernels take them.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
_MIN_NORMAL_EXP = -6          # smallest normal: 2^-6
_MANT_BITS = 3


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """float64 values of e4m3 codes (NaN patterns decode to NaN)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = sign * np.ldexp(1.0 + m / 8.0, e - 7)
    sub = sign * np.ldexp(m / 8.0, _MIN_NORMAL_EXP)
    v = np.where(e == 0, sub, normal)
    return np.where((e == 15) & (m == 7), np.nan, v)


def e4m3_encode_rne(v: np.ndarray) -> np.ndarray:
    """Nearest e4m3 code to each float (float32 or float64 values), ties to even mantissa,
    magnitudes above 448 saturated to 448."""
    v = np.asarray(v, dtype=np.float64)
    neg = np.signbit(v)
    a = np.minimum(np.abs(v), E4M3_MAX)
    # quantum of the binade (subnormals share the smallest normal binade's quantum 2^-9)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, _MIN_NORMAL_EXP)
    q = np.ldexp(1.0, (e - _MANT_BITS).astype(np.int64))
    r = np.rint(a / q) * q                      # np.rint rounds half to even
    r = np.minimum(r, E4M3_MAX)
    # encode the rounded magnitude (it may have moved up a binade)
    with np.errstate(divide="ignore"):
        er = np.floor(np.log2(np.where(r > 0, r, 1.0)))
    is_sub = r < np.ldexp(1.0, _MIN_NORMAL_EXP)
    exp_field = np.where(is_sub, 0, er + 7).astype(np.int64)
    mant = np.where(is_sub, r / np.ldexp(1.0, _MIN_NORMAL_EXP - _MANT_BITS),
                    r / np.ldexp(1.0, (er - _MANT_BITS).astype(np.int64)) - 8.0)
    code = (exp_field << 3) | np.rint(mant).astype(np.int64)
    code = np.where(r == 0, 0, code)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


def quantize_rows_e4m3(rows: np.ndarray):
    """Per-row scaling and e4m3 codes of a [n, width] array of exact fp32 values (bf16 inputs).

    Returns (codes uint8 [n, width], scales float32 [n])."""
    v = np.asarray(rows, dtype=np.float32)
    amax = np.max(np.abs(v), axis=1) if v.shape[1] else np.zeros(v.shape[0], np.float32)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    scaled = (v / scale[:, None]).astype(np.float32)   # fp32 division, round to nearest
    return e4m3_encode_rne(scaled), scale


def dequantize_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """float64 values the quantised rows stand for: code value times the row's scale (exact)."""
    return e4m3_decode(codes) * np.asarray(scales, np.float64)[:, None]


def gate_up_fp8(xq: np.ndarray, xs: np.ndarray, gq: np.ndarray, gs: np.ndarray, uq: np.ndarray,
                us: np.ndarray) -> np.ndarray:
    """h = silu(a) * b for quantised rows: a = (s_x q_x) (s_g q_g)^T, b likewise with the up rows,
    in float64.  xq [n, d] codes, xs [n]; gq, uq [f, d] codes, gs, us [f] (one expert)."""
    x = dequantize_rows(xq, xs)
    a = x @ dequantize_rows(gq, gs).T
    b = x @ dequantize_rows(uq, us).T
    return a / (1.0 + np.exp(-a)) * b
