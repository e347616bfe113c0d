"""Pins for the oracle's FP4 E2M1 format, NVFP4 Q/K quantizer and its attention mode (CPU only).

NVFP4 ("VisualGen Quantized Attention", section "MXFP8 and NVFP4 in the CUTEDSL and FlashInfer
backends": Q/K in fixed blocks of 16 elements, V in FP8) is read as NVIDIA's two-level format: E2M1
elements, an unsigned E4M3 scale per block of 16 channels, a float32 scale per tensor. Pins, none of
which re-types the oracle's formula:

* E2M1: every code's value from its bit fields (bias 1, one mantissa bit), a hand table of
  roundings (all ties, saturation, signed zero), monotonicity and the half-gap bound;
* nibble packing order on a hand case;
* hand-derived blocks (tensor scale 2688 / amax, block bytes and codes worked out by hand),
  a layout check whose block bytes follow in closed form (block max 6 * 2^e -> byte 126 + 8e), the
  zero block, and invariance of codes and bytes under power-of-two scaling of the tensor;
* block-scaled BMM1 = the product of the dequantized operands; the attention equals QK16PV8 over
  the dequantized Q/K; Q = 0 gives uniform attention (LSE = ln Skv).
"""

import math

import numpy as np
import pytest

from oracle import attention as att
from oracle import formats
from oracle import nvfp4_quant
from oracle import sage_quant


def test_e2m1_values_from_bit_fields():
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
        assert formats.e2m1_decode(code) == (-mag if s else mag)
        assert formats.e2m1_encode(formats.e2m1_decode(code)) == code  # -0 included


# value -> code; ties go to the even code (even mantissa bit)
E2M1_CASES = [(0.0, 0), (-0.0, 8), (0.1, 0), (-0.1, 8), (0.25, 0), (0.26, 1), (0.5, 1), (0.75, 2), (1.0, 2),
              (1.25, 2), (1.26, 3), (1.75, 4), (2.5, 4), (2.51, 5), (3.0, 5), (3.5, 6), (4.9, 6), (5.0, 6),
              (5.01, 7), (6.0, 7), (7.0, 7), (1e30, 7), (-2.5, 12), (-3.5, 14), (-100.0, 15)]


@pytest.mark.parametrize("x,code", E2M1_CASES)
def test_e2m1_rounding_table(x, code):
    assert int(formats.e2m1_encode(np.float32(x))) == code


def test_e2m1_monotone_and_within_half_gap():
    x = np.linspace(-7, 7, 20001).astype(np.float32)
    v = formats.e2m1_decode(formats.e2m1_encode(x))
    assert np.all(np.diff(v) >= 0)
    grid = formats.E2M1_VALUES
    gaps = np.diff(grid)
    a = np.minimum(np.abs(x), 6.0)
    i = np.clip(np.searchsorted(grid, a, side="right") - 1, 0, len(gaps) - 1)
    assert np.all(np.abs(np.abs(v) - a) <= gaps[i] / 2 + 1e-12)


def test_nibble_packing_order():
    assert formats.pack_nibbles(np.array([1, 2, 3, 4, 15, 0], np.uint8)).tolist() == [0x21, 0x43, 0x0F]
    assert formats.unpack_nibbles(np.array([0x21, 0xF0], np.uint8)).tolist() == [1, 2, 0, 15]


def _tensor(blocks):
    """[1, 1, 1, 128] tensor whose 16-channel blocks start with the given values."""
    x = np.zeros((1, 1, 1, 128), np.float32)
    for c, vals in enumerate(blocks):
        x[0, 0, 0, 16 * c:16 * c + len(vals)] = vals
    return x


def test_hand_derived_blocks():
    # tensor amax 6: S = 2688 / 6 = 448.
    # block 0 amax 6: 6 / 6 * 448 = 448 -> byte 0x7E; factor 448 / 448 = 1: 6 -> 7, 3 -> 5, -1.5 -> 0xB, 0.25 -> 0 (tie)
    # block 1 amax 0.75: 0.125 * 448 = 56 = 1.75 * 2^5 -> byte 0x66; factor 448 / 56 = 8:
    #   0.75 -> 6 -> 7, 0.3 -> 2.4 -> 2 (code 4), -0.1 -> -0.8 -> -1 (0xA), 0.0625 -> 0.5 (code 1)
    # block 2 zero: byte 0, codes 0
    x = _tensor([[6.0, 3.0, -1.5, 0.25], [0.75, 0.3, -0.1, 0.0625]])
    packed, sf, S = nvfp4_quant.nvfp4_quantize(x)
    assert S == np.float32(448.0)
    assert sf[0, 0, 0].tolist() == [0x7E, 0x66, 0, 0, 0, 0, 0, 0]
    codes = formats.unpack_nibbles(packed)[0, 0, 0]
    assert codes[:4].tolist() == [7, 5, 0xB, 0]
    assert codes[16:20].tolist() == [7, 4, 0xA, 1]
    assert not codes[4:16].any() and not codes[20:].any()


def test_all_zero_tensor():
    packed, sf, S = nvfp4_quant.nvfp4_quantize(np.zeros((1, 3, 2, 128), np.float32))
    assert S == 1.0 and not packed.any() and not sf.any()


def test_block_bytes_follow_the_block_max_in_head_major_layout():
    # one tensor-wide max of 6 (S = 448) in head 0; block (b, t, h, c) holds 6 * 2^e with e in [-10, -1], whose
    # byte is E4M3(2^e * 448) = E4M3(1.75 * 2^(8 + e)) = 0x7E + 8e, and whose element encodes to 6 (code 7);
    # the other heads' maxima are below 6, so a scale taken per head would change their bytes
    B, T, H = 2, 5, 3
    x = np.zeros((B, T, H, 128), np.float32)
    want = np.zeros((B, H, T, 8), np.int64)
    for b in range(B):
        for t in range(T):
            for h in range(H):
                for c in range(8):
                    e = -1 - (3 * b + 5 * t + 7 * h + c) % 10
                    x[b, t, h, 16 * c + (t + c) % 16] = np.float32(6.0 * 2.0 ** e)
                    want[b, h, t, c] = 0x7E + 8 * e
    x[0, 0, 0, 0] = 6.0  # the tensor max (its block's byte is then 0x7E whatever e was)
    want[0, 0, 0, 0] = 0x7E
    packed, sf, S = nvfp4_quant.nvfp4_quantize(x)
    assert S == np.float32(448.0)
    assert np.array_equal(sf.astype(np.int64), want)
    codes = formats.unpack_nibbles(packed)
    assert np.all(codes[x != 0] == 7) and np.all(codes[x == 0] == 0)


def test_power_of_two_scaling_of_the_tensor_changes_only_its_scale():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((1, 7, 3, 128)).astype(np.float32)
    packed, sf, S = nvfp4_quant.nvfp4_quantize(x)
    for k in (-12, -1, 3, 20):
        p2, s2, S2 = nvfp4_quant.nvfp4_quantize((x * np.float32(2.0 ** k)).astype(np.float32))
        assert np.array_equal(p2, packed) and np.array_equal(s2, sf)
        assert S2 == np.float32(S * 2.0 ** -k)


def test_round_trip_error_is_within_the_block_bound():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((2, 64, 2, 128)) * np.exp(rng.uniform(-3, 3, (2, 64, 2, 8))).repeat(16, axis=3))
    x = x.astype(np.float32)
    packed, sf, S = nvfp4_quant.nvfp4_quantize(x)
    deq = nvfp4_quant.nvfp4_decode(packed, sf, S)
    amax = np.abs(x.reshape(2, 64, 2, 8, 16)).max(axis=4).repeat(16, axis=3)
    # half the widest E2M1 gap (1, between 4 and 6) of the block scale amax / 6, widened by the E4M3
    # rounding of that scale (2^-4), plus what saturation can cut off when the scale rounds down
    assert np.all(np.abs(deq - x) <= amax * ((1 + 2.0 ** -4) / 6 + 2.0 ** -4) + 1e-30)


def test_scores_equal_the_product_of_dequantized_operands():
    rng = np.random.default_rng(3)
    q = (rng.standard_normal((1, 40, 1, 128)) * np.exp(rng.uniform(-2, 2, (1, 40, 1, 128)))).astype(np.float32)
    k = (rng.standard_normal((1, 70, 1, 128)) * np.exp(rng.uniform(-2, 2, (1, 70, 1, 128)))).astype(np.float32)
    qc, qs, qS = nvfp4_quant.nvfp4_quantize(q)
    kc, ks, kS = nvfp4_quant.nvfp4_quantize(k)
    got = nvfp4_quant.nvfp4_scores(qc[0, :, 0], qs[0, 0], qS, kc[0, :, 0], ks[0, 0], kS)
    want = nvfp4_quant.nvfp4_decode(qc, qs, qS)[0, :, 0] @ nvfp4_quant.nvfp4_decode(kc, ks, kS)[0, :, 0].T
    assert np.max(np.abs(got - want) / (np.abs(want) + 1e-30)) < 1e-12


def test_attention_is_qk16pv8_attention_of_the_dequantized_q_and_k():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 200, 2, 128)).astype(np.float32)
    k = (rng.standard_normal((1, 260, 1, 128)) * 3).astype(np.float32)
    v = rng.standard_normal((1, 260, 1, 128)).astype(np.float32)
    quant = nvfp4_quant.nvfp4_qk_quantize(q, k, v, per_tensor=True)
    deq = dict(q=nvfp4_quant.nvfp4_decode(quant["q_codes"], quant["q_sf"], quant["q_gs"]),
               k=nvfp4_quant.nvfp4_decode(quant["k_codes"], quant["k_sf"], quant["k_gs"]), v=v)
    ref = sage_quant.qk16pv8_quantize(v, True)
    for h in range(2):
        for t in range(2):
            o, _, _, lse = att.attention_q_tile(dict(q=q, k=k, v=v), 0, h, t, mode="nvfp4", quant=quant,
                                                with_lse=True)
            o2, _, _, lse2 = att.attention_q_tile(deq, 0, h, t, mode="qk16pv8", quant=ref, with_lse=True)
            assert np.max(np.abs(o - o2)) < 1e-9 and np.max(np.abs(lse - lse2)) < 1e-12


def test_q_zero_is_uniform_attention():
    rng = np.random.default_rng(5)
    Skv = 333
    q = np.zeros((1, 128, 1, 128), np.float32)
    k = rng.standard_normal((1, Skv, 1, 128)).astype(np.float32)
    v = rng.standard_normal((1, Skv, 1, 128)).astype(np.float32)
    quant = nvfp4_quant.nvfp4_qk_quantize(q, k, v, False)
    o, _, _, lse = att.attention_q_tile(dict(q=q, k=k, v=v), 0, 0, 0, mode="nvfp4", quant=quant, with_lse=True)
    assert np.max(np.abs(lse - math.log(Skv))) < 1e-12
    vdeq = formats.e4m3_decode(quant["v_codes"][0, :, 0]) * quant["v_scale"][0, 0][None, :]
    assert np.max(np.abs(o - vdeq.mean(axis=0)[None, :])) < 1e-12


def test_nvfp4_is_a_coarser_approximation_of_dense_attention():
    # sanity only: 4-bit Q/K on top of QK16PV8's FP8 P.V
    rng = np.random.default_rng(6)
    q = rng.standard_normal((1, 128, 1, 128)).astype(np.float32)
    k = rng.standard_normal((1, 256, 1, 128)).astype(np.float32)
    v = rng.standard_normal((1, 256, 1, 128)).astype(np.float32)
    quant = nvfp4_quant.nvfp4_qk_quantize(q, k, v, False)
    o, _, _ = att.attention_q_tile(dict(q=q, k=k, v=v), 0, 0, 0, mode="nvfp4", quant=quant)
    dense = att.dense_attention(q, k, v)[0, :, 0]
    assert np.linalg.norm(o - dense) / np.linalg.norm(dense) < 0.3
