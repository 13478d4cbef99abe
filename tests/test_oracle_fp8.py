"""Pins of the oracle's FP8 (e4m3) quantisation step (CPU)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8


def test_decode_landmarks():
    v = fp8.e4m3_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x39, 0x7E, 0xFE, 0x80], np.uint8))
    assert list(v) == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.125, 448.0, -448.0, 0.0]
    assert np.isnan(fp8.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    assert np.array_equal(fp8.e4m3_encode_rne(fp8.e4m3_decode(codes)), codes)


def test_ties_go_to_even_and_large_values_saturate():
    v = np.array([1.0625, 1.1875, 2.0 ** -9 * 0.5, 2.0 ** -9 * 1.5, 464.0, 1000.0, -1000.0])
    got = fp8.e4m3_decode(fp8.e4m3_encode_rne(v))
    assert list(got) == [1.0, 1.25, 0.0, 2.0 * 2.0 ** -9, 448.0, 448.0, -448.0]


def test_matches_torch_float8_conversion():
    # an independent implementation of the same rounding (round to nearest even, in range)
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1e-2, 20000),
                        rng.normal(0, 1, 20000)]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode_rne(v), ref)


def test_row_scaling_uses_the_whole_range():
    rng = np.random.default_rng(1)
    rows = rng.normal(0, 3, (64, 200)).astype(np.float32)
    q, s = fp8.quantize_rows_e4m3(rows)
    dec = fp8.e4m3_decode(q)
    assert np.all(np.abs(dec).max(axis=1) == 448.0)
    # relative error of every element within half an e4m3 step of its binade (2^-4), plus the
    # subnormal floor
    err = np.abs(dec * s[:, None] - rows)
    assert np.all(err <= np.abs(rows) * 2.0 ** -4 + s[:, None] * 2.0 ** -10)
    z, zs = fp8.quantize_rows_e4m3(np.zeros((2, 8), np.float32))
    assert not z.any() and np.all(zs == 1.0)


def test_lossless_inputs_reduce_to_the_bf16_expert():
    # values already on the e4m3 grid, with row maxima 448 * 2^j: quantisation is exact, so the
    # quantised projection equals the plain expert forward's h on the same values
    rng = np.random.default_rng(2)
    grid = fp8.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    grid = grid[grid >= 2.0 ** -3]

    def rows(n, w, j):
        r = rng.choice(grid, (n, w)) * rng.choice([-1.0, 1.0], (n, w))
        r[:, 0] = 448.0
        return (r * 2.0 ** j).astype(np.float32)
    x, wg, wu = rows(5, 64, -6), rows(32, 64, -9), rows(32, 64, -9)
    xq, xs = fp8.quantize_rows_e4m3(x)
    gq, gs = fp8.quantize_rows_e4m3(wg)
    uq, us = fp8.quantize_rows_e4m3(wu)
    h = fp8.gate_up_fp8(xq, xs, gq, gs, uq, us)
    _, _, h_ref, _ = oracle.expert_forward(x.astype(np.float64), wg.astype(np.float64),
                                           wu.astype(np.float64), np.zeros((1, 32)))
    assert np.allclose(h, h_ref, rtol=1e-12, atol=0)
