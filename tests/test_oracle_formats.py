"""Pins for the oracle's number formats (E2M1, E4M3, NVFP4 packing, activation rule).

Each test checks the oracle against something other than itself: the format
definitions written out as closed-form value lists, torch's float8_e4m3fn
decoder (a library routine), and exhaustive midpoint / saturation cases.
"""
import numpy as np
import pytest
import torch

from oracle import formats as F


def test_e2m1_table_closed_form():
    # E2M1 magnitudes: 0, 0.5 (subnormal), then (1 + m/2) * 2^(e-1) for e = 1..3
    assert list(F.E2M1_TABLE[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(F.E2M1_TABLE[8:]) == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e4m3_table_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.E4M3_TABLE
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all() and nan.sum() == 2          # 0x7F and 0xFF
    assert (ours[~nan] == ref[~nan]).all()
    assert np.nanmax(ours) == 448.0 and F.E4M3_TABLE[1] == 2.0 ** -9


def test_encode_decode_identity_on_all_codes():
    for c in range(16):
        v = F.E2M1_TABLE[c]
        if c == 8:   # -0 encodes with its sign bit
            assert F.e2m1_encode(np.array([-0.0]))[0] == 8
            continue
        assert F.e2m1_encode(np.array([v]))[0] == c
    for c in range(256):
        v = F.E4M3_TABLE[c]
        if np.isnan(v) or c == 0x80:
            continue
        assert F.e4m3_encode(np.array([v]))[0] == c, c


@pytest.mark.parametrize("table,enc,n", [(F.E2M1_TABLE, F.e2m1_encode, 8),
                                          (F.E4M3_TABLE, F.e4m3_encode, 127)])
def test_rne_midpoints_and_neighbours(table, enc, n):
    pos = table[:n]
    for i in range(n - 1):
        a, b = pos[i], pos[i + 1]
        mid = (a + b) / 2
        even = i if i % 2 == 0 else i + 1
        assert enc(np.array([mid]))[0] == even
        assert enc(np.array([-mid]))[0] == even | (8 if n == 8 else 0x80)
        assert enc(np.array([np.nextafter(mid, 0)]))[0] == i
        assert enc(np.array([np.nextafter(mid, np.inf)]))[0] == i + 1


def test_saturation():
    assert F.E2M1_TABLE[F.e2m1_encode(np.array([6.0, 7.0, 1e30, -1e30]))].tolist() == [6, 6, 6, -6]
    assert F.E4M3_TABLE[F.e4m3_encode(np.array([448.0, 460.0, 1e9, -1e9]))].tolist() == [448, 448, 448, -448]


def test_e4m3_encode_matches_torch_in_range():
    # torch's fp32 -> float8_e4m3fn conversion rounds to nearest-even in range
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(20000) * 30, rng.uniform(-2 ** -6, 2 ** -6, 5000)])
    v = v[np.abs(v) < 448].astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = F.e4m3_encode(v)
    ok = (ours == ref) | ((ours & 0x7F) == 0) & ((ref & 0x7F) == 0)
    assert ok.all()


def test_nvfp4_unpack_low_nibble_first():
    codes = np.array([[0x21, 0xF7]], dtype=np.uint8)
    assert F.nvfp4_unpack_codes(codes).tolist() == [[1, 2, 7, 15]]
    deq = F.nvfp4_dequantize(np.tile(codes, (1, 4)), np.array([[0x38]], np.uint8), 2.0)  # block scale 1.0
    assert deq[0, :4].tolist() == [1.0, 2.0, 12.0, -12.0]


def test_activation_rule_representable_roundtrip():
    # rows built as e2m1 * e4m3 * s with the block max at magnitude 6 and the row max
    # block scale at 448 reproduce exactly
    rng = np.random.default_rng(2)
    q = rng.integers(0, 16, size=(4, 64))
    q[:, ::16] = 7                       # each block holds a 6
    sc = rng.integers(0x20, 0x60, size=(4, 4))
    sc[:, 0] = 0x7E                      # 448 in the first block of each row
    s = np.array([0.5, 1.0, 2.0 ** -7, 3.0])
    v = F.E2M1_TABLE[q] * np.repeat(F.E4M3_TABLE[sc], 16, axis=1) * s[:, None]
    q2, sc2, s2 = F.quantize_activation(v)
    assert np.array_equal(F.dequantize_activation(q2, sc2, s2), v)
    assert np.array_equal(s2, s.astype(np.float32))


def test_activation_rule_error_bound_and_zero_rows():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((16, 256)) * np.exp(rng.uniform(-8, 8, size=(16, 1)))
    v[3] = 0.0
    deq = F.fake_quantize_activation(v)
    amax_b = np.repeat(np.abs(v).reshape(16, 16, 16).max(axis=2), 16, axis=1)
    # one E2M1 step is at most 2 units of the block scale (~amax_b/6), plus E4M3 rounding
    assert (np.abs(deq - v) <= amax_b * (1.0 / 6.0) * (1 + 2 ** -3) + 1e-300).all()
    assert (deq[3] == 0).all()
    # scale-1 rows (the SwiGLU output between the expert GEMMs)
    deq1 = F.fake_quantize_activation(v / np.maximum(np.abs(v).max(axis=1, keepdims=True), 1e-30), row_scale=False)
    assert np.isfinite(deq1).all()
