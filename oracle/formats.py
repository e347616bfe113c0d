"""8-bit code formats used by SAGE quantization (oracle side; test infrastructure only).

FP8 E4M3 is the format the pages name for SAGE Q/K ("fp8_e4m3") and for V, which "is
always quantized per channel to FP8 E4M3" ("TRTLLM Attention" user guide, section "SAGE
quantization"). INT8 is the other Q/K option there. The pages give neither bit layout
nor rounding rule, so these readings apply (each is pinned in tests/test_oracle_formats.py; the
FP4 E2M1 element type of NVFP4 is defined with its encoder below):

* E4M3 is the "fn" variant: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
  no infinities, a single NaN mantissa pattern (S.1111.111), largest finite 448,
  smallest normal 2^-6, subnormal step 2^-9. Conversion rounds to nearest, ties to even
  mantissa, and saturates every magnitude above 448 to 448 (``satfinite``). The sign of
  a value that rounds to zero is kept (code 0x80 for negative zero).
* INT8 is symmetric: code = clamp(round_half_even(x), -127, 127); -128 is never produced.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
INT8_MAX = 127.0
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_SUBNORMAL_STEP = 2.0 ** -9


def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 bit pattern (uint8) as float64; the NaN pattern decodes to NaN."""
    c = np.asarray(codes).astype(np.uint8)
    sign = (c >> 7) & 1
    exp = ((c >> 3) & 0xF).astype(np.int64)
    man = (c & 0x7).astype(np.float64)
    normal = (1.0 + man / 8.0) * np.exp2(exp - 7.0)
    subnormal = man * E4M3_SUBNORMAL_STEP
    val = np.where(exp == 0, subnormal, normal)
    val = np.where((exp == 15) & (man == 7), np.nan, val)
    return np.where(sign == 1, -val, val)


def e4m3_encode(x) -> np.ndarray:
    """Round real values (given as float32 or float64) to E4M3 codes (uint8).

    Round to nearest, ties to even; magnitudes above 448 saturate to 448; NaN maps to the
    NaN pattern. Works on the exact value it is given, so a float32 input is rounded once.
    Large arrays are encoded in slices (element by element, so the result is the same).
    """
    x = np.asarray(x)
    if x.size > (1 << 24):
        flat = x.reshape(-1)
        out = np.empty(flat.shape, dtype=np.uint8)
        for s0 in range(0, flat.size, 1 << 24):
            out[s0:s0 + (1 << 24)] = _e4m3_encode_slice(flat[s0:s0 + (1 << 24)])
        return out.reshape(x.shape)
    return _e4m3_encode_slice(x)


def _e4m3_encode_slice(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    with np.errstate(divide="ignore", invalid="ignore"):
        # Subnormal range (and zero): integer multiples of 2^-9; 8 * 2^-9 is the smallest
        # normal, whose code (0b0001000) continues the subnormal codes without a gap.
        sub_code = np.rint(np.minimum(a, E4M3_MIN_NORMAL) / E4M3_SUBNORMAL_STEP)
        # Normal range: a = f * 2^E with f in [0.5, 1) -> unbiased exponent e = E - 1,
        # mantissa steps of 2^(e-3), so a / 2^(e-3) lies in [8, 16).
        _, E = np.frexp(a)
        e = E.astype(np.int64) - 1
        q = np.rint(np.ldexp(a, (3 - e)))
        carry = q >= 16.0
        e = np.where(carry, e + 1, e)
        q = np.where(carry, 8.0, q)
        biased = e + 7
        normal_code = (biased << 3) | (q.astype(np.int64) - 8)
    code = np.where(a < E4M3_MIN_NORMAL, sub_code.astype(np.int64), normal_code)
    # Saturation: anything beyond the largest finite value (code 0x7E = 448) clamps to it.
    code = np.where((a > E4M3_MAX) | (code > 0x7E), 0x7E, code)
    code = np.where(nan, 0x7F, code)
    code = np.where(neg, code | 0x80, code)
    return code.astype(np.uint8)


# FP4 E2M1 (the NVFP4 element type): 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit; the
# eight magnitudes of codes 0..7, no infinities or NaN. Largest finite 6, subnormal 0.5.
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
E2M1_MAX = 6.0


def e2m1_encode(x) -> np.ndarray:
    """Round real values to E2M1 codes (uint8 in 0..15, sign in bit 3).

    Round to nearest, ties to the even code (even mantissa bit); magnitudes above 6 saturate to
    6; the sign of a value that rounds to zero is kept (code 8 for negative zero).
    """
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.minimum(np.abs(x), E2M1_MAX)
    d = np.abs(a[..., None] - E2M1_VALUES)                 # exact for float32 / float64 inputs
    best = d.min(axis=-1, keepdims=True)
    cand = d == best                                        # one code, or two adjacent ones on a tie
    even = cand & (np.arange(8) % 2 == 0)
    code = np.where(even.any(axis=-1), np.argmax(even, axis=-1), np.argmax(cand, axis=-1))
    return np.where(neg, code | 8, code).astype(np.uint8)


def e2m1_decode(codes) -> np.ndarray:
    """Value of each E2M1 code (0..15) as float64."""
    c = np.asarray(codes).astype(np.int64)
    val = E2M1_VALUES[c & 7]
    return np.where(c & 8, -val, val)


def pack_nibbles(codes) -> np.ndarray:
    """Pack 4-bit codes along the last axis two per byte: element 2i in bits 0-3, 2i+1 in bits 4-7."""
    c = np.asarray(codes).astype(np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed) -> np.ndarray:
    """Inverse of ``pack_nibbles``."""
    p = np.asarray(packed).astype(np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def int8_code(x) -> np.ndarray:
    """Symmetric INT8 code of float32 values: round half to even, clamp to [-127, 127]."""
    x = np.asarray(x, dtype=np.float32)
    return np.clip(np.rint(x), -INT8_MAX, INT8_MAX).astype(np.int8)


def code_values(codes, qk_dtype: str) -> np.ndarray:
    """Float64 value of a code array: INT8 codes are integers, E4M3 codes decode."""
    if qk_dtype == "int8":
        return np.asarray(codes).astype(np.float64)
    if qk_dtype == "fp8_e4m3":
        return e4m3_decode(codes)
    raise ValueError(f"unknown code dtype {qk_dtype!r}")
