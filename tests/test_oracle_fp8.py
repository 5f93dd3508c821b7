"""Pins for the oracle's FP8 E4M3 decoder (CPU)."""
import numpy as np
import torch

from oracle import dequant, e4m3_to_float64


def test_format_values():
    # values the E4M3 "fn" format fixes: bias 7, 3 mantissa bits, max 448, NaN code
    cases = {0x00: 0.0, 0x38: 1.0, 0x40: 2.0, 0x3C: 1.5, 0x7E: 448.0, 0x08: 2.0 ** -6,
             0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0xB8: -1.0, 0xFE: -448.0, 0x80: -0.0}
    for code, v in cases.items():
        assert e4m3_to_float64(np.array([code]))[0] == v, hex(code)
    assert np.isnan(e4m3_to_float64(np.array([0x7F, 0xFF]))).all()


def test_all_codes_match_library_decoder():
    codes = np.arange(256, dtype=np.uint8)
    ours = e4m3_to_float64(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    same = (ours == lib) | (np.isnan(ours) & np.isnan(lib))
    assert same.all(), codes[~same]


def test_positive_codes_increase():
    v = e4m3_to_float64(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(v) > 0)


def test_dequant_uses_the_fp32_scale():
    s = 0.1  # not representable: the fp32 rounding of 0.1 is the cache's scale
    y = dequant(np.array([0x38]), s)
    assert y[0] == float(np.float32(0.1))
