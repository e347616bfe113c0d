"""Planted mistakes: each test swaps a plausible bug into the oracle (on the CPU, through
monkeypatch) and checks that at least one pin then fails. This is what gives the pins
their meaning: a dropped term, a wrong sign, index or rounding rule must not pass."""

import numpy as np
import pytest

from oracle import attention as att
from oracle import formats, sage_quant

from . import test_oracle_attention as TA
from . import test_oracle_formats as TF
from . import test_oracle_lse as TLSE
from . import test_oracle_quant as TQ
from . import test_oracle_sage_lossless as TL


def _fails(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def test_round_half_away_in_e4m3_is_caught(monkeypatch):
    good = formats.e4m3_encode

    def half_away(x):
        x = np.asarray(x, np.float64)
        # nudge exact ties upward in magnitude before rounding (round half away from zero)
        return good(x * (1 + 2.0 ** -30))
    monkeypatch.setattr(formats, "e4m3_encode", half_away)
    _fails(TF.test_e4m3_encoder_exhaustive_bf16_vs_brute_force)


def test_truncating_int8_is_caught(monkeypatch):
    monkeypatch.setattr(formats, "int8_code",
                        lambda x: np.clip(np.trunc(np.asarray(x, np.float32)), -127, 127).astype(np.int8))
    _fails(TF.test_int8_half_even_and_clamp)


def test_quotient_losing_the_sign_of_zero_is_caught(monkeypatch):
    # -0 + 0 = +0: a quotient formed through a sum with a positive zero encodes -0 as 0x00
    good = sage_quant._codes_from_quotient
    monkeypatch.setattr(sage_quant, "_codes_from_quotient",
                        lambda quot, dtype: good(np.asarray(quot, np.float32) + np.float32(0.0), dtype))
    _fails(TQ.test_negative_zero_keeps_its_sign_in_e4m3_codes)


def test_k_mean_over_s_minus_one_is_caught(monkeypatch):
    def biased(k):
        k = np.asarray(k, np.float32)
        return (k.astype(np.float64).sum(axis=1) / (k.shape[1] - 1)).astype(np.float32)
    monkeypatch.setattr(sage_quant, "k_channel_mean", biased)
    _fails(TQ.test_k_mean_constant_channel_is_exact)


def test_lse_in_base_two_is_caught(monkeypatch):
    good = att.dense_lse
    monkeypatch.setattr(att, "dense_lse", lambda q, k, rows=None: good(q, k, rows) / np.log(2.0))
    _fails(TLSE.test_tiled_lse_equals_logsumexp_of_brute_force_logits, 128)


def test_block_absmax_over_all_heads_is_caught(monkeypatch):
    good = sage_quant.quantize_token_blocks

    def all_heads(x, block, qk_dtype):
        # one scale per token block shared by every head: the head axis taken into the block max
        x = np.asarray(x, np.float32)
        _, scales = good(x, block, qk_dtype)
        scales = np.broadcast_to(scales.max(axis=1, keepdims=True), scales.shape).copy()
        row_scale = np.repeat(scales, block, axis=2)[:, :, :x.shape[1]].transpose(0, 2, 1)[:, :, :, None]
        with np.errstate(divide="ignore", invalid="ignore"):
            quot = np.where(row_scale == 0, np.float32(0), (x / row_scale).astype(np.float32))
        return sage_quant._codes_from_quotient(quot, qk_dtype), scales
    monkeypatch.setattr(sage_quant, "quantize_token_blocks", all_heads)
    _fails(TQ.test_block_quant_matches_brute_force, "int8", 4)


def test_smoothed_q_is_caught(monkeypatch):
    good = sage_quant.sage_quantize

    def q_smoothed(q, k, v, qk_dtype, q_block, k_block, k_mean=None):
        out = good(q, k, v, qk_dtype, q_block, k_block, k_mean)
        qs = sage_quant.smooth_k(q, out["k_mean"])  # Hq == Hkv in the pin
        out["q_codes"], out["q_scale"] = sage_quant.quantize_token_blocks(qs, q_block, qk_dtype)
        return out
    monkeypatch.setattr(sage_quant, "sage_quantize", q_smoothed)
    _fails(TQ.test_q_is_not_smoothed, "int8")


def test_missing_k_smoothing_is_caught(monkeypatch):
    monkeypatch.setattr(sage_quant, "smooth_k", lambda k, mean: np.asarray(k, np.float32))
    _fails(TQ.test_smoothed_k_has_zero_channel_mean)


def test_wrong_qmax_is_caught(monkeypatch):
    monkeypatch.setitem(sage_quant.QMAX, "int8", np.float32(128.0))
    _fails(TQ.test_constant_block_gives_full_scale_codes, "int8", 4)


def test_dropped_softmax_scale_is_caught(monkeypatch):
    monkeypatch.setattr(att, "SOFTMAX_SCALE", 1.0)
    _fails(TA.test_dense_matches_scalar_brute_force)


def test_wrong_gqa_mapping_is_caught(monkeypatch):
    monkeypatch.setattr(att, "kv_head_of", lambda hq, Hq, Hkv: hq % Hkv)
    _fails(TA.test_gqa_equals_mha_with_replicated_kv)


def test_transposed_value_operand_is_caught(monkeypatch):
    good = att.dense_attention

    def transposed(q, k, v, rows=None):
        v = np.asarray(v, np.float64)
        return good(q, k, v[:, :, :, ::-1], rows)
    monkeypatch.setattr(att, "dense_attention", transposed)
    _fails(TA.test_dense_matches_scalar_brute_force)


def test_missing_online_rescale_is_caught(monkeypatch):
    def no_alpha(s, values, *, quantize_p, threshold=None):
        rows, skv = s.shape
        m = np.full(rows, -np.inf)
        l = np.zeros(rows)
        acc = np.zeros((rows, values.shape[1]))
        for t0 in range(0, skv, att.TILE):
            st = s[:, t0:t0 + att.TILE]
            m_new = np.maximum(m, st.max(axis=1))
            p = np.exp(st - m_new[:, None])
            l = l + p.sum(axis=1)                      # bug: no alpha
            acc = acc + p @ values[t0:t0 + att.TILE]
            m = m_new
        return acc / l[:, None], 0
    monkeypatch.setattr(att, "tiled_attention", no_alpha)
    _fails(TA.test_tiled_loop_equals_untiled_definition)


def test_skip_rule_with_wrong_sign_is_caught(monkeypatch):
    good = att.tiled_attention

    def wrong_sign(s, values, *, quantize_p, threshold=None):
        # bug: compares exp(m_run - m_tile) instead of exp(m_tile - m_run)
        return good(-s, values, quantize_p=quantize_p, threshold=threshold)
    monkeypatch.setattr(att, "tiled_attention", wrong_sign)
    _fails(TA.test_skip_matches_prefix_max_closed_form, 200.0)


def test_wrong_p_scale_is_caught(monkeypatch):
    monkeypatch.setattr(formats, "E4M3_MAX", 256.0)
    _fails(TA.test_sage_single_tile_formula, "int8")


# ---- QK16PV8 (V in FP8 with a tensor-wide or per-channel scale, BF16 Q/K)
from . import test_oracle_qk16pv8 as TP  # noqa: E402


def test_channel_max_used_as_tensor_scale_is_caught(monkeypatch):
    monkeypatch.setattr(sage_quant, "quantize_v_per_tensor", sage_quant.quantize_v_per_channel)
    _fails(TP.test_tensor_scale_closed_form_and_extreme_code)


def test_unquantized_p_in_qk16pv8_is_caught(monkeypatch):
    good = att.tiled_attention
    monkeypatch.setattr(att, "tiled_attention",
                        lambda s, values, quantize_p, threshold=None, with_lse=False:
                        good(s, values, quantize_p=False, threshold=threshold, with_lse=with_lse))
    _fails(TP.test_one_row_matches_scalar_definition)


def test_dropped_v_scale_in_qk16pv8_is_caught(monkeypatch):
    good = sage_quant.qk16pv8_quantize

    def unit_scale(v, per_tensor):
        res = good(v, per_tensor)
        res["v_scale"] = np.ones_like(res["v_scale"])
        return res
    monkeypatch.setattr(sage_quant, "qk16pv8_quantize", unit_scale)
    _fails(TP.test_large_logits_give_the_target_value_row, True)


# ---- MXFP8 Q/K (block-32 E4M3 elements with E8M0 scales)
from oracle import mx_quant  # noqa: E402

from . import test_oracle_mx as TM  # noqa: E402


def test_scale_rounded_up_instead_of_floor_rule_is_caught(monkeypatch):
    # the no-saturation variant: 2^ceil(log2(amax / 448)) instead of 2^(floor(log2 amax) - 8)
    def ceil_rule(amax):
        a = np.asarray(amax, np.float64)
        with np.errstate(divide="ignore"):
            e = np.ceil(np.log2(a / 448.0))
        return np.clip(np.where(a == 0, -127, e), -127, 127).astype(np.int64)
    monkeypatch.setattr(mx_quant, "shared_exponent", ceil_rule)
    _fails(TM.test_hand_derived_blocks, [1.9375, 1.0], 119, [0x7E, 0x78])


def test_off_by_one_element_emax_is_caught(monkeypatch):
    monkeypatch.setattr(mx_quant, "E4M3_EMAX", 7)
    _fails(TM.test_hand_derived_blocks, [3.0, -3.0, 0.0], 120, [0x7C, 0xFC, 0x00])


def test_token_major_scale_layout_is_caught(monkeypatch):
    good = mx_quant.mx_quantize

    def token_major(x):
        codes, sf = good(x)
        return codes, np.ascontiguousarray(sf.transpose(0, 2, 1, 3))
    monkeypatch.setattr(mx_quant, "mx_quantize", token_major)
    _fails(TM.test_every_block_has_its_own_scale_in_head_major_layout)


def test_one_block_scale_for_all_blocks_is_caught(monkeypatch):
    def first_block_scale(qc, qs, kc, ks):
        qs = np.repeat(np.asarray(qs)[:, :1], 4, axis=1)
        ks = np.repeat(np.asarray(ks)[:, :1], 4, axis=1)
        a, b = formats.e4m3_decode(qc), formats.e4m3_decode(kc)
        return (a @ b.T) * np.ldexp(1.0, qs[:, 0].astype(np.int64) - 127)[:, None] \
            * np.ldexp(1.0, ks[:, 0].astype(np.int64) - 127)[None, :]
    monkeypatch.setattr(mx_quant, "mx_scores", first_block_scale)
    _fails(TM.test_mx_scores_equal_the_product_of_dequantized_operands)


def test_unquantized_q_k_in_mxfp8_attention_is_caught(monkeypatch):
    good = att.attention_q_tile

    def dense_logits(inputs, b, hq, tile, **kw):
        if kw.get("mode") == "mxfp8":
            kw = dict(kw, mode="qk16pv8")
        return good(inputs, b, hq, tile, **kw)
    monkeypatch.setattr(att, "attention_q_tile", dense_logits)
    _fails(TM.test_mxfp8_attention_is_qk16pv8_attention_of_the_dequantized_q_and_k)


# ---- NVFP4 Q/K (E2M1 elements, E4M3 block scales per 16 channels, float32 tensor scale)
from oracle import nvfp4_quant  # noqa: E402

from . import test_oracle_nvfp4 as TN  # noqa: E402


def test_swapped_nibble_order_is_caught(monkeypatch):
    monkeypatch.setattr(formats, "pack_nibbles",
                        lambda c: (np.asarray(c, np.uint8)[..., 1::2] | (np.asarray(c, np.uint8)[..., 0::2] << 4)))
    _fails(TN.test_nibble_packing_order)


def test_e2m1_ties_away_from_zero_is_caught(monkeypatch):
    good = formats.e2m1_encode
    monkeypatch.setattr(formats, "e2m1_encode", lambda x: good(np.asarray(x, np.float64) * (1 + 2.0 ** -30)))
    _fails(TN.test_e2m1_rounding_table, 2.5, 4)


def test_per_head_tensor_scale_is_caught(monkeypatch):
    good = nvfp4_quant.nvfp4_quantize

    def per_head(x, scale=None):
        outs = [good(x[:, :, h:h + 1]) for h in range(x.shape[2])]
        packed = np.concatenate([o[0] for o in outs], axis=2)
        sf = np.concatenate([o[1] for o in outs], axis=1)
        return packed, sf, outs[0][2]
    monkeypatch.setattr(nvfp4_quant, "nvfp4_quantize", per_head)
    _fails(TN.test_block_bytes_follow_the_block_max_in_head_major_layout)


def test_missing_tensor_scale_is_caught(monkeypatch):
    monkeypatch.setattr(nvfp4_quant, "tensor_scale", lambda x: np.float32(1.0))
    _fails(TN.test_hand_derived_blocks)


def test_sage_dropped_k_scale_is_caught(monkeypatch):
    good = att.sage_scores
    monkeypatch.setattr(att, "sage_scores", lambda qc, kc, qs, ks, dt: good(qc, kc, qs, np.ones_like(ks), dt))
    _fails(TL._compare, "int8", 1, 16, None)


def test_sage_k_scale_of_the_next_block_is_caught(monkeypatch):
    good = att.sage_scores
    monkeypatch.setattr(att, "sage_scores", lambda qc, kc, qs, ks, dt: good(qc, kc, qs, np.roll(ks, -16), dt))
    _fails(TL._compare, "fp8_e4m3", 1, 16, None)


def test_sage_q_scale_of_the_previous_row_is_caught(monkeypatch):
    good = att.sage_scores
    monkeypatch.setattr(att, "sage_scores", lambda qc, kc, qs, ks, dt: good(qc, kc, np.roll(qs, 1), ks, dt))
    _fails(TL._compare, "int8", 4, 4, None)


def test_code_dots_in_float32_are_caught(monkeypatch):
    # float32 accumulation: exact for INT8 codes (sums below 2^22) but not for E4M3 products
    monkeypatch.setattr(att, "code_dots", lambda qc, kc, dt: (formats.code_values(qc, dt).astype(np.float32) @
                                                              formats.code_values(kc, dt).astype(np.float32).T
                                                              ).astype(np.float64))
    _fails(TA.test_code_dot_products_match_triple_loop)


def test_wrong_e2m1_value_is_caught(monkeypatch):
    table = np.array(formats.E2M1_VALUES, dtype=np.float64)
    table[7] = 5.0  # the largest magnitude taken as 5 instead of 6
    monkeypatch.setattr(formats, "E2M1_VALUES", table)
    _fails(TN.test_e2m1_values_from_bit_fields)


def test_mx_decode_with_the_wrong_bias_is_caught(monkeypatch):
    good = mx_quant.mx_decode
    monkeypatch.setattr(mx_quant, "mx_decode", lambda codes, sf: good(codes, sf) * 2.0)  # bias 126 in decode only
    _fails(TM.test_round_trip_error_is_within_e4m3_rounding)


def test_nvfp4_scores_with_the_neighbouring_block_scale_are_caught(monkeypatch):
    good = nvfp4_quant.nvfp4_scores
    monkeypatch.setattr(nvfp4_quant, "nvfp4_scores", lambda qc, qsf, qs, kc, ksf, ks:
                        good(qc, qsf, qs, kc, np.roll(np.asarray(ksf), 1, axis=-1), ks))
    _fails(TN.test_scores_equal_the_product_of_dequantized_operands)


def test_swapped_nibbles_on_unpacking_are_caught(monkeypatch):
    good = formats.unpack_nibbles

    def swapped(p):
        out = good(p)
        return np.stack([out[..., 1::2], out[..., 0::2]], axis=-1).reshape(out.shape)
    monkeypatch.setattr(formats, "unpack_nibbles", swapped)
    _fails(TN.test_nibble_packing_order)

