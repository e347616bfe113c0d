"""Pins for the oracle's MXFP8 Q/K quantizer and its attention mode (CPU only).

The quantizer follows the OCP Microscaling (MX) v1.0 definition of MXFP8 with E4M3 elements,
block 32 along the head dimension ("VisualGen Quantized Attention", section "MXFP8 and NVFP4 in
the CUTEDSL and FlashInfer backends": fixed blocks of 32 elements; cuDNN section: block scaling
along the head dimension). Pins, none of which re-types the oracle's formula:

* hand-derived cases from the format's definition (shared exponent floor(log2 amax) - 8, E8M0
  byte = exponent + 127, E4M3 element codes including saturation, the zero block and both
  ends of the E8M0 range);
* invariants: scaling a block by 2^k moves its byte by k and leaves its codes; every block is
  scaled on its own (a layout check with distinct exponents per token, head and block);
* the E4M3 rounding bound on the round trip;
* BMM1 on MX operands equals the product of the dequantized operands, and on inputs that MXFP8
  represents exactly the whole MXFP8 attention equals QK16PV8 (same V path) bit for bit;
* closed form Q = 0: uniform attention (LSE = ln Skv).
"""

import math

import numpy as np
import pytest

from oracle import attention as att
from oracle import formats
from oracle import mx_quant
from oracle import sage_quant


def _one_block(values):
    x = np.zeros((1, 1, 1, 128), np.float32)
    x[0, 0, 0, :len(values)] = np.asarray(values, np.float32)
    codes, sf = mx_quant.mx_quantize(x)
    return codes[0, 0, 0, :len(values)], int(sf[0, 0, 0, 0]), sf[0, 0, 0, 1:]


# (block values, expected E8M0 byte, expected E4M3 codes); derivations:
#   amax 3 = 1.5 * 2^1: exponent 1 - 8 = -7 -> byte 120; 3 / 2^-7 = 384 = 1.5 * 2^8 -> E4M3 0x7C
#   amax 1: exponent -8 -> byte 119; 256 -> 0x78; 0.5 -> 128 -> 0x70; -0.25 -> -64 -> 0xE8 (exp 13)
#   amax 0.875 = 1.75 * 2^-1: exponent -9 -> byte 118; 448 -> 0x7E (largest finite)
#   amax 1.9375: exponent -8 -> byte 119; 496 > 448 saturates to 0x7E; 1.0 -> 256 -> 0x78
#   amax 2^-130 (a bfloat16 subnormal): exponent -138 clamps to -127 -> byte 0; 2^-3 -> 0x20
#   amax 2^127: exponent 119 -> byte 246; 256 -> 0x78
#   the zero block: byte 0 and zero codes
CASES = [
    ([3.0, -3.0, 0.0], 120, [0x7C, 0xFC, 0x00]),
    ([1.0, 0.5, -0.25], 119, [0x78, 0x70, 0xE8]),
    ([0.875, 0.4375], 118, [0x7E, 0x76]),
    ([1.9375, 1.0], 119, [0x7E, 0x78]),
    ([2.0 ** -130], 0, [0x20]),
    ([2.0 ** 127, -(2.0 ** 126)], 246, [0x78, 0xF0]),
    ([0.0, -0.0], 0, [0x00, 0x80]),
]


@pytest.mark.parametrize("values,byte,codes", CASES)
def test_hand_derived_blocks(values, byte, codes):
    got_codes, got_byte, other = _one_block(values)
    assert got_byte == byte
    assert got_codes.tolist() == codes
    assert other.tolist() == [0, 0, 0]  # the other three blocks of the token are zero


def test_scaling_a_block_by_a_power_of_two_moves_only_its_byte():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((1, 3, 2, 128)).astype(np.float32)
    codes, sf = mx_quant.mx_quantize(x)
    for k in (-20, -1, 1, 7, 40):
        y = (x * np.float32(2.0 ** k)).astype(np.float32)
        c2, s2 = mx_quant.mx_quantize(y)
        assert np.array_equal(c2, codes)
        assert np.array_equal(s2.astype(np.int64), sf.astype(np.int64) + k)


def test_every_block_has_its_own_scale_in_head_major_layout():
    B, S, H = 2, 5, 3
    x = np.zeros((B, S, H, 128), np.float32)
    want = np.zeros((B, H, S, 4), np.int64)
    for b in range(B):
        for t in range(S):
            for h in range(H):
                for c in range(4):
                    e = (7 * b + 5 * t + 3 * h + c) % 23 - 11
                    x[b, t, h, 32 * c + (t + c) % 32] = np.float32(2.0 ** e)  # the block's only nonzero
                    want[b, h, t, c] = e - 8 + 127
    codes, sf = mx_quant.mx_quantize(x)
    assert np.array_equal(sf.astype(np.int64), want)
    assert np.all(codes[x != 0] == 0x78) and np.all(codes[x == 0] == 0)


def test_round_trip_error_is_within_e4m3_rounding():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((2, 64, 2, 128)) * np.exp(rng.uniform(-6, 6, (2, 64, 2, 1)))).astype(np.float32)
    codes, sf = mx_quant.mx_quantize(x)
    deq = mx_quant.mx_decode(codes, sf)
    e = sf.astype(np.int64).transpose(0, 2, 1, 3) - 127
    X = np.repeat(np.ldexp(1.0, e), 32, axis=3)            # [B, S, H, 128]
    q = np.abs(x.astype(np.float64)) / X
    err = np.abs(deq - x)
    normal = (q >= 2.0 ** -6) & (q <= 448)
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(x[normal]) + 1e-300)
    assert np.all(err[q < 2.0 ** -6] <= 2.0 ** -10 * X[q < 2.0 ** -6])
    sat = q > 448
    assert np.all(np.abs(deq[sat]) == 448 * X[sat])
    assert np.all(q < 512)                                 # amax / X < 2^9 by construction


def test_mx_scores_equal_the_product_of_dequantized_operands():
    rng = np.random.default_rng(3)
    q = (rng.standard_normal((1, 40, 1, 128)) * np.exp(rng.uniform(-3, 3, (1, 40, 1, 128)))).astype(np.float32)
    k = (rng.standard_normal((1, 70, 1, 128)) * np.exp(rng.uniform(-3, 3, (1, 70, 1, 128)))).astype(np.float32)
    qc, qs = mx_quant.mx_quantize(q)
    kc, ks = mx_quant.mx_quantize(k)
    got = mx_quant.mx_scores(qc[0, :, 0], qs[0, 0], kc[0, :, 0], ks[0, 0])
    want = mx_quant.mx_decode(qc, qs)[0, :, 0] @ mx_quant.mx_decode(kc, ks)[0, :, 0].T
    assert np.max(np.abs(got - want) / (np.abs(want) + 1e-30)) < 1e-12


def _exact_inputs(rng, shape):
    """Values that MXFP8 holds exactly: per (token, head, block) a power of two times elements
    from {0, +-0.5, ..., +-1.75}, whose E4M3 images are exact and never saturate."""
    base = np.array([0, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, -0.5, -0.75, -1.0, -1.25, -1.5, -1.75])
    B, S, H, D = shape
    vals = rng.choice(base, size=shape)
    e = rng.integers(-4, 4, size=(B, S, H, 4))
    return (vals * np.repeat(np.ldexp(1.0, e), 32, axis=3)).astype(np.float32)


def test_exactly_representable_inputs_give_the_qk16pv8_result_bit_for_bit():
    rng = np.random.default_rng(4)
    q = _exact_inputs(rng, (1, 130, 2, 128))
    k = _exact_inputs(rng, (1, 300, 1, 128))
    v = rng.standard_normal((1, 300, 1, 128)).astype(np.float32)
    quant = mx_quant.mxfp8_quantize(q, k, v, per_tensor=False)
    assert np.array_equal(mx_quant.mx_decode(quant["q_codes"], quant["q_sf"]), q)
    ref = sage_quant.qk16pv8_quantize(v, False)
    inp = dict(q=q, k=k, v=v)
    for h in range(2):
        for t in range(2):
            o, _, _, lse = att.attention_q_tile(inp, 0, h, t, mode="mxfp8", quant=quant, with_lse=True)
            o2, _, _, lse2 = att.attention_q_tile(inp, 0, h, t, mode="qk16pv8", quant=ref, with_lse=True)
            assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_mxfp8_attention_is_qk16pv8_attention_of_the_dequantized_q_and_k():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 200, 2, 128)).astype(np.float32)
    k = (rng.standard_normal((1, 260, 1, 128)) * 3).astype(np.float32)
    v = rng.standard_normal((1, 260, 1, 128)).astype(np.float32)
    quant = mx_quant.mxfp8_quantize(q, k, v, per_tensor=True)
    deq = dict(q=mx_quant.mx_decode(quant["q_codes"], quant["q_sf"]), k=mx_quant.mx_decode(quant["k_codes"], quant["k_sf"]),
               v=v)
    assert not np.array_equal(deq["q"], q)  # the inputs are not exactly representable
    ref = sage_quant.qk16pv8_quantize(v, True)
    for h in range(2):
        for t in range(2):
            o, _, _, lse = att.attention_q_tile(dict(q=q, k=k, v=v), 0, h, t, mode="mxfp8", quant=quant,
                                                with_lse=True)
            o2, _, _, lse2 = att.attention_q_tile(deq, 0, h, t, mode="qk16pv8", quant=ref, with_lse=True)
            assert np.max(np.abs(o - o2)) < 1e-9 and np.max(np.abs(lse - lse2)) < 1e-12


def test_q_zero_is_uniform_attention():
    rng = np.random.default_rng(5)
    Skv = 333
    q = np.zeros((1, 128, 1, 128), np.float32)
    k = rng.standard_normal((1, Skv, 1, 128)).astype(np.float32)
    v = rng.standard_normal((1, Skv, 1, 128)).astype(np.float32)
    for per_tensor in (False, True):
        quant = mx_quant.mxfp8_quantize(q, k, v, per_tensor)
        assert np.all(quant["q_sf"] == 0) and np.all(quant["q_codes"] == 0)
        o, _, _, lse = att.attention_q_tile(dict(q=q, k=k, v=v), 0, 0, 0, mode="mxfp8", quant=quant, with_lse=True)
        assert np.max(np.abs(lse - math.log(Skv))) < 1e-12
        vdeq = formats.e4m3_decode(quant["v_codes"][0, :, 0]) * quant["v_scale"][0, 0][None, :]
        assert np.max(np.abs(o - vdeq.mean(axis=0)[None, :])) < 1e-12  # p = 1 is exact in E4M3


def test_mxfp8_is_close_to_dense_attention():
    # sanity only: the error of 8-bit Q/K on top of QK16PV8's FP8 P.V (about 3.5% here)
    rng = np.random.default_rng(6)
    q = rng.standard_normal((1, 128, 1, 128)).astype(np.float32)
    k = rng.standard_normal((1, 256, 1, 128)).astype(np.float32)
    v = rng.standard_normal((1, 256, 1, 128)).astype(np.float32)
    quant = mx_quant.mxfp8_quantize(q, k, v, False)
    o, _, _ = att.attention_q_tile(dict(q=q, k=k, v=v), 0, 0, 0, mode="mxfp8", quant=quant)
    dense = att.dense_attention(q, k, v)[0, :, 0]
    assert np.linalg.norm(o - dense) / np.linalg.norm(dense) < 0.1
