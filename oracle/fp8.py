"""TEST INFRASTRUCTURE ONLY: exact decoding of FP8 e4m3 codes to float64.

e4m3 (the "FN" variant used for FP8 Q K^T, named among FlashAttention's
production modes in "GPU Kernels: CUDA, HIP & Triton", section 7.6): 1 sign
bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities; exponent
field 0 is subnormal (value m/8 * 2^-6), and the single code with all
exponent and mantissa bits set is NaN.  Every finite code is exactly a
float64, so the oracle consumes the decoded values without rounding.
"""
from __future__ import annotations

import numpy as np


def decode_e4m3(codes) -> np.ndarray:
    """uint8 e4m3 codes (any shape) -> float64 values, by the definition."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = sign * np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    subnormal = sign * np.ldexp(m / 8.0, -6)
    out = np.where(e == 0, subnormal, normal)
    return np.where((e == 0xF) & (m == 0x7), np.nan, out)
