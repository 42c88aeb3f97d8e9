"""Rounding of float64 values to the storage types the operators emit (oracle; test infrastructure).

The operator pages fix the output dtypes (MlaPrologV2 README, "参数说明": BF16 / FLOAT16 / INT8
outputs; aclnnQkvRmsNormRopeCache, "Formulas" (4): int8 quantised caches) but not the rounding
rule.  The reading used throughout: round to nearest, ties to even (IEEE 754 default), for the
floating formats; round half to even then saturate for int8.

The float formats are written from their definitions, not through any library cast:
a binary format with p significand bits (implicit bit included), minimum normal exponent emin and
maximum exponent emax represents x as an integer multiple of 2^(max(e, emin) - (p-1)), where
2^e <= |x| < 2^(e+1).  Rounding x is rounding x / quantum to the nearest integer (ties to even).
"""
from __future__ import annotations

import numpy as np


def _round_binary(x, p: int, emin: int, emax: int) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        _, e = np.frexp(x)                     # x = m * 2^e with 0.5 <= |m| < 1
        exp = np.maximum(e - 1, emin)          # exponent of the leading bit, clamped at emin
        quantum_exp = exp - (p - 1)
        y = np.ldexp(np.rint(np.ldexp(x, -quantum_exp)), quantum_exp)
        largest = (2.0 - 2.0 ** (1 - p)) * 2.0 ** emax
        y = np.where(np.abs(y) > largest, np.copysign(np.inf, x), y)
        y = np.where(np.isfinite(x), y, x)     # inf and nan pass through
    return y


def round_bf16(x) -> np.ndarray:
    """Nearest bfloat16 value (8 significand bits, exponent range of binary32)."""
    return _round_binary(x, p=8, emin=-126, emax=127)


def round_fp16(x) -> np.ndarray:
    """Nearest IEEE binary16 value (11 significand bits, emin -14, emax 15)."""
    return _round_binary(x, p=11, emin=-14, emax=15)


def round_fp32(x) -> np.ndarray:
    """Nearest IEEE binary32 value (24 significand bits, emin -126, emax 127)."""
    return _round_binary(x, p=24, emin=-126, emax=127)


def saturate_int8_rne(v, lo: int = -128, hi: int = 127) -> np.ndarray:
    """Round half to even, then clamp to [lo, hi]; returned as int8."""
    v = np.asarray(v, dtype=np.float64)
    return np.clip(np.rint(v), lo, hi).astype(np.int8)
