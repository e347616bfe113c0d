"""Pins for the oracle's 8-bit code formats (CPU only).

The E4M3 encoder is checked against things that do not share its arithmetic: the format's
closed-form special values, a brute-force nearest-value search over the 127 positive
finite codes (ties to the even code), and PyTorch's float8_e4m3fn cast. The INT8 rounding
is checked on its half-way cases and clamp.
"""

import numpy as np
import pytest
import torch

from oracle import formats


def test_e4m3_closed_form_values():
    d = formats.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert d[0x00] == 0.0 and d[0x80] == 0.0 and np.signbit(d[0x80])
    assert d[0x01] == 2.0 ** -9                 # smallest subnormal
    assert d[0x07] == 7 * 2.0 ** -9             # largest subnormal
    assert d[0x08] == 2.0 ** -6                 # smallest normal
    assert d[0x38] == 1.0                       # exponent field 7 = bias
    assert d[0x7E] == 448.0                     # largest finite
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF])
    assert d[0xBE] == -1.75                     # sign 1, exponent 7, mantissa 6/8
    # strictly increasing over the positive finite codes
    pos = d[:0x7F]
    assert np.all(np.diff(pos) > 0)
    assert np.array_equal(d[0x80:0xFF], -pos)


def _brute_force_nearest(x: np.ndarray) -> np.ndarray:
    """Nearest positive finite E4M3 value by exhaustive search; ties go to the even code."""
    table = formats.e4m3_decode(np.arange(0x7F, dtype=np.uint8))  # codes 0..0x7E
    a = np.abs(x.astype(np.float64))
    dist = np.abs(a[:, None] - table[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    codes = np.arange(0x7F)
    # among tied candidates pick the even code (RNE); at most two candidates tie
    even = cand & (codes[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), np.argmax(even, axis=1), np.argmax(cand, axis=1))
    pick = np.where(a > 448.0, 0x7E, pick)
    return np.where(np.signbit(x), pick | 0x80, pick).astype(np.uint8)


def _all_finite_bf16() -> np.ndarray:
    bits = np.arange(65536, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    return x[np.isfinite(x)]


def test_e4m3_encoder_exhaustive_bf16_vs_brute_force():
    x = _all_finite_bf16()
    got = formats.e4m3_encode(x)
    want = _brute_force_nearest(x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first x={x[bad[:5]]} got={got[bad[:5]]} want={want[bad[:5]]}"


def test_e4m3_encoder_random_fp32_vs_brute_force():
    rng = np.random.default_rng(7)
    # magnitudes spread over the whole code range, including subnormals and saturation
    x = (rng.standard_normal(200_000) * np.exp2(rng.uniform(-14, 10, 200_000))).astype(np.float32)
    got = formats.e4m3_encode(x)
    assert np.array_equal(got, _brute_force_nearest(x))


def test_e4m3_encoder_matches_torch_cast_in_range():
    x = _all_finite_bf16()
    x = x[np.abs(x) <= 448.0]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(formats.e4m3_encode(x), want)


def test_e4m3_ties_and_saturation():
    cases = {
        1.0625: 0x38,           # halfway between 1.0 (even) and 1.125 -> 1.0
        1.1875: 0x3A,           # halfway between 1.125 and 1.25 (even) -> 1.25
        2.0 ** -10: 0x00,       # half the smallest subnormal -> 0 (even)
        3 * 2.0 ** -10: 0x02,   # halfway 1 and 2 subnormal steps -> 2 (even)
        448.0: 0x7E,
        464.0: 0x7E,            # halfway to the (unrepresentable) 480 -> saturates
        1e30: 0x7E,
        -1e30: 0xFE,
        -1e-9: 0x80,            # negative value rounding to zero keeps its sign
    }
    for x, code in cases.items():
        assert formats.e4m3_encode(np.float32(x)) == code, x
    assert formats.e4m3_encode(np.float32(np.nan)) == 0x7F


def test_e4m3_roundtrip_of_representable_values():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = formats.e4m3_decode(codes)
    assert np.array_equal(formats.e4m3_encode(vals), codes)


def test_int8_half_even_and_clamp():
    x = np.array([0.5, -0.5, 1.5, -1.5, 2.5, -2.5, 126.5, 127.4, 127.6, 200.0, -200.0, -127.5], np.float32)
    want = np.array([0, 0, 2, -2, 2, -2, 126, 127, 127, 127, -127, -127], np.int8)
    assert np.array_equal(formats.int8_code(x), want)
    assert formats.int8_code(np.float32(-128.0)) == -127    # -128 is never produced


@pytest.mark.parametrize("dtype", ["int8", "fp8_e4m3"])
def test_code_values(dtype):
    if dtype == "int8":
        c = np.arange(-127, 128).astype(np.int8)
        assert np.array_equal(formats.code_values(c, dtype), np.arange(-127, 128))
    else:
        assert formats.code_values(np.uint8(0x7E), dtype) == 448.0
