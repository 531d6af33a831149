"""Pins for the FP8 E4M3 oracle: the format's defining values, agreement with
PyTorch's float8_e4m3fn conversions (a library routine) on every code and on
every in-range bf16 value, ties to even, saturation, and the round trip."""
import numpy as np
import pytest
import torch

from oracle import quant as Q


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x38, 1.0), (0xB8, -1.0), (0x7E, 448.0), (0xFE, -448.0), (0x01, 2.0 ** -9),
    (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6), (0x3C, 1.5), (0x40, 2.0), (0x30, 0.5), (0x77, 240.0),
])
def test_defining_values(code, value):
    assert Q.e4m3_to_f64(np.array([code], dtype=np.uint8))[0] == value


def test_nan_and_negative_zero():
    v = Q.e4m3_to_f64(np.array([0x7F, 0xFF, 0x80], dtype=np.uint8))
    assert np.isnan(v[0]) and np.isnan(v[1]) and v[2] == 0.0 and np.signbit(v[2])


def test_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = Q.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(ours[~both_nan], ref[~both_nan]) and np.array_equal(np.isnan(ours), np.isnan(ref))


def test_encode_matches_torch_on_all_in_range_bf16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    keep = np.isfinite(vals) & (np.abs(vals) <= 448.0)
    vals = vals[keep]
    ours = Q.f64_to_e4m3(vals.astype(np.float64))
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_ties_to_even_and_saturation():
    c = Q.f64_to_e4m3(np.array([1.0625, 1.1875, 1000.0, -1e30, 449.0, 2.0 ** -10, 3 * 2.0 ** -11, np.nan]))
    v = Q.e4m3_to_f64(c)
    assert v[0] == 1.0 and v[1] == 1.25                    # midpoints go to the even mantissa
    assert v[2] == 448.0 and v[3] == -448.0 and v[4] == 448.0
    assert v[5] == 0.0                                      # half of the smallest subnormal: tie to even (0)
    assert v[6] == 2.0 ** -9                                # 0.75 * 2^-9 -> nearest subnormal 2^-9
    assert np.isnan(v[7])


def test_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(Q.f64_to_e4m3(Q.e4m3_to_f64(codes)), codes)


def test_quantize_uses_float32_division():
    x = np.array([1.0, -3.0, 0.3, 1e-3], dtype=np.float32)
    s = np.float32(0.1)
    want = Q.f64_to_e4m3((x / s).astype(np.float64))
    assert np.array_equal(Q.quantize(x, s), want)
    np.testing.assert_array_equal(Q.dequantize(Q.quantize(x, s), s),
                                  Q.e4m3_to_f64(want) * float(s))
    # An input whose float32 quotient is exactly the midpoint 1.0625 of the
    # codes for 1.0 (even) and 1.125 (odd) while the exact quotient lies
    # above it: a float32 division rounds it to 1.0 (tie to the even code),
    # a float64 one to 1.125.
    x0 = np.float32(1.0625 * float(s))
    pick = None
    for k in range(-64, 65):
        xc = np.float32(x0 + np.float32(k) * np.spacing(x0))
        if np.float32(xc) / s == np.float32(1.0625) and float(xc) / float(s) > 1.0625:
            pick = xc
            break
    assert pick is not None
    assert Q.e4m3_to_f64(Q.quantize(np.array([pick], dtype=np.float32), s))[0] == 1.0
    assert Q.e4m3_to_f64(Q.f64_to_e4m3(np.array([float(pick) / float(s)])))[0] == 1.125
