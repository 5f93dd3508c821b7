"""FP8 E4M3 decoding for the oracle (test infrastructure).

The pages list an fp8 KV cache among the untested variants ("vLLM's custom ROCm
paged-attention kernel wins all sixty cells", §6). The cache format used here is
the E4M3 "fn" encoding of the OCP 8-bit floating-point standard: 1 sign bit, 4
exponent bits with bias 7, 3 mantissa bits; exponent 0 holds subnormals
(m/8 * 2^-6); there are no infinities and S.1111.111 is NaN; the largest finite
magnitude is 448. A cache element decodes to code_value * scale, with one fp32
scale per tensor (K and V separately). Attention over the decoded K/V is then the
ordinary definition in decode_ref.
"""
from __future__ import annotations

import numpy as np


def e4m3_to_float64(codes: np.ndarray) -> np.ndarray:
    """Decode uint8 E4M3 codes to float64, exactly."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = (c >> 7) & 1
    exp = (c >> 3) & 0xF
    man = c & 0x7
    normal = (1.0 + man / 8.0) * np.power(2.0, exp - 7)
    subnormal = (man / 8.0) * 2.0 ** -6
    val = np.where(exp == 0, subnormal, normal)
    val = np.where((exp == 0xF) & (man == 0x7), np.nan, val)
    return np.where(sign == 1, -val, val)


def dequant(codes: np.ndarray, scale: float) -> np.ndarray:
    """Cache value of each code: e4m3(code) * scale (scale widened from fp32)."""
    return e4m3_to_float64(codes) * float(np.float32(scale))
